// Decode step for small units: one consumer warp per unit.
//
// Computes exactly what k_decode does for a unit -- GQA attention over the
// retained tokens, the importance update imp_j += sum_h p_hj (blog sec. 3
// "H2O"; HiKV Stage I's recent-bank rule when enabled), the argmin victim,
// and in a fused step the append and the one-token eviction -- but with a
// whole unit in one warp.  Ragged per-head budgets (HeadKV summary sec. 3.2)
// leave most units with a few hundred tokens; for those the CTA-wide merge,
// the barriers and the cluster exchanges of k_decode cost as much as the
// tile loop.  Here a unit needs no barrier beyond its warp:
//   producer warp   lane w streams the tiles of warp w's units into the two
//                   ring stages {w, w + 4} that only warp w consumes, and
//                   their q (and new rows) into warp w's double buffer;
//   consumer warp w the tile loop of k_decode (row-split q.k with q in
//                   registers, lazily rescaled online softmax, lane-owns-dims
//                   p.v), then the output,
//                   the importance pass over the logits it kept in shared
//                   memory, the victim by warp shuffles, and the fused move.
// Units come from a per-warp list the host balances (largest first to the
// least-loaded warp).
#pragma once

#include "k_decode.cuh"

namespace hikv {

constexpr int kSmallThreads = (kSmallWarps + 1) * 32;
constexpr int kSmallMaxPg = 32;                         // page ids cached per warp

template <typename T, int D, int G>
struct SmallLayout {
    static constexpr int RB = D * (int)sizeof(T);
    static constexpr int TB = kDecTR * RB;
    static constexpr int QB = G * D * (int)sizeof(T);
    static constexpr int STAGES = 2 * kSmallWarps;
    static constexpr int RING = 0;                                            // [STAGES][2 TB]
    static constexpr int BARS = RING + STAGES * 2 * TB;                       // full, empty [STAGES]; qfull, qempty [W][2]
    static constexpr int QRAW = BARS + (2 * STAGES + 4 * kSmallWarps) * 8;    // [W][2][QB]
    static constexpr int NROW = QRAW + kSmallWarps * 2 * QB;                  // [W][2][2 RB]
    static constexpr int QS = NROW + kSmallWarps * 2 * 2 * RB;                // [W][G D] f32
    static constexpr int PS = QS + kSmallWarps * G * D * 4;                   // [W][16][G] f32
    static constexpr int S = PS + kSmallWarps * kDecTR * G * 4;               // [W][kSmallLogitFloats] f32
    static constexpr int PG = S + kSmallWarps * kSmallLogitFloats * 4;        // [W][kSmallMaxPg] i32
    static constexpr int TOTAL = PG + kSmallWarps * kSmallMaxPg * 4 + 1024;   // + base alignment slack
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(kSmallThreads, 2)
    k_decode_small(const SmallArgs a, const __grid_constant__ CUtensorMap tmap) {
    using Lay = SmallLayout<T, D, G>;
    constexpr int ESZ = (int)sizeof(T);
    constexpr int RB = Lay::RB, TB = Lay::TB, QB = Lay::QB;
    constexpr int EPL = D / 32, LB = EPL * ESZ;
    constexpr int NCAP = small_unit_cap(G);
    // row-split q.k, as in k_decode: QK_LPR lanes per row, one 16-byte chunk
    // each against q in registers; per sub-block of QK_SUB warp steps the
    // QK_NV (row, head) partial sums are reduce-scattered over the row's lanes
    constexpr int QK_LPR = RB / 16;
    constexpr int QK_RPW = 32 / QK_LPR;
    constexpr int QK_STEPS = kDecTR / QK_RPW;
    constexpr int QK_EPL = 16 / ESZ;
    constexpr int QK_SUB = (QK_LPR / G) > QK_STEPS ? QK_STEPS : (QK_LPR / G);
    constexpr int QK_NSUB = QK_STEPS / QK_SUB;
    constexpr int QK_NV = QK_SUB * G;
    constexpr int QK_DUP = QK_LPR / QK_NV;
    static_assert(EPL % 2 == 0 && QK_EPL % 2 == 0, "pairs");
    static_assert(QK_SUB >= 1 && QK_STEPS % QK_SUB == 0 && QK_LPR % QK_NV == 0, "one logit per lane and sub-block");
    using Raw = typename RawVec<LB>::type;

    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const View& v = a.v;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint8_t* ring = smem + Lay::RING;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::BARS);
    uint64_t* empty = full + Lay::STAGES;
    uint64_t* qfull = empty + Lay::STAGES;        // [W][2]
    uint64_t* qempty = qfull + 2 * kSmallWarps;   // [W][2]

    if (tid == 0) {
        for (int s = 0; s < Lay::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2 * kSmallWarps; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();
    const int32_t per_layer = v.batch * v.hkv;

    if (warp == kSmallWarps) {
        // ======================= producer: lane w feeds warp w =======================
        if (lane < kSmallWarps) {
            const int w = lane;
            const int wi = blockIdx.x * kSmallWarps + w;
            const int32_t i0 = a.warp_off[wi], i1 = a.warp_off[wi + 1];
            int32_t* pg_s = reinterpret_cast<int32_t*>(smem + Lay::PG) + w * kSmallMaxPg;
            int gj = 0;   // tiles issued for warp w so far
            bool ok = true;
            for (int k = 0; ok && i0 + k < i1; ++k) {
                const int32_t u = a.list[i0 + k];
                const int32_t n = v.len[u] + a.fused;
                const int32_t li = u / per_layer - a.layer0, b = (u / v.hkv) % v.batch, g = u % v.hkv;
                const int qb = k & 1;
                if (!mbar_wait_bounded(&qempty[w * 2 + qb], ((uint32_t)(k >> 1) & 1u) ^ 1u, v.err, kWaitQEmpty,
                                       (uint32_t)k)) {
                    ok = false;
                    break;
                }
                const int64_t qoff = ((((int64_t)li * v.batch + b) * v.hq + (int64_t)g * G) * D) * ESZ;
                mbar_arrive_expect_tx(&qfull[w * 2 + qb], QB + (a.fused ? 2 * RB : 0));
                bulk_g2s(smem + Lay::QRAW + (w * 2 + qb) * QB, a.q + qoff, QB, &qfull[w * 2 + qb]);
                if (a.fused) {
                    const int64_t ui = (int64_t)u - (int64_t)a.layer0 * per_layer;
                    uint8_t* nr = smem + Lay::NROW + (w * 2 + qb) * 2 * RB;
                    bulk_g2s(nr, a.new_k + ui * RB, RB, &qfull[w * 2 + qb]);
                    bulk_g2s(nr + RB, a.new_v + ui * RB, RB, &qfull[w * 2 + qb]);
                }
                const int32_t nt = ceil_div(n, kDecTR);
                const int32_t npg = ceil_div(n, v.page_tokens);
                const int32_t* ptab = v.page_table + (int64_t)u * v.max_pages;
                for (int j = 0; j < min(npg, kSmallMaxPg); ++j) pg_s[j] = ptab[j];
                for (int32_t i = 0; i < nt; ++i, ++gj) {
                    const int st = w + kSmallWarps * (gj & 1);
                    if (!mbar_wait_bounded(&empty[st], ((uint32_t)(gj >> 1) & 1u) ^ 1u, v.err, kWaitEmpty,
                                           (uint32_t)gj)) {
                        ok = false;
                        break;
                    }
                    const int32_t s0 = i * kDecTR;
                    const int32_t pi = s0 >> v.page_shift;
                    const int32_t pg = pi < kSmallMaxPg ? pg_s[pi] : ptab[pi];
                    if (pg < 0 || pg >= v.pool_pages) {
                        atomicOr(v.err, DEVERR_PAGE);
                        mbar_arrive(&full[st]);   // complete the stage without data
                        ok = false;
                        ++gj;
                        break;
                    }
                    uint8_t* dst = ring + st * 2 * TB;
                    mbar_arrive_expect_tx(&full[st], 2 * TB);
                    dec_load_tile<true, 1, ESZ, RB, TB>(dst, v, pg, s0, &tmap, &full[st]);
                }
            }
            if (!ok) {
                // let this lane's copies in flight land before the CTA can exit
                for (int j = max(0, gj - 2); j < gj; ++j)
                    mbar_wait_bounded(&full[w + kSmallWarps * (j & 1)], (uint32_t)(j >> 1) & 1u, v.err, kWaitDrain,
                                      (uint32_t)j);
            }
        }
        __syncwarp();
        __syncthreads();
        return;
    }

    // ======================= consumer warp: one unit at a time =======================
    const int wi = blockIdx.x * kSmallWarps + warp;
    const int32_t i0 = a.warp_off[wi], i1 = a.warp_off[wi + 1];
    float* q_s = reinterpret_cast<float*>(smem + Lay::QS) + warp * G * D;
    float* ps = reinterpret_cast<float*>(smem + Lay::PS) + warp * kDecTR * G;
    float* S = reinterpret_cast<float*>(smem + Lay::S) + warp * kSmallLogitFloats;
    const int qk_c = lane % QK_LPR, qk_rg = lane / QK_LPR;
    const int qk_k = qk_c / QK_DUP, qk_step = qk_k / G, hk = qk_k % G;
    const bool qk_own = (qk_c % QK_DUP) == 0;
    const int pv_chunk = (lane * LB) >> 4, pv_in = (lane * LB) & 15;
    int gj = 0;
    bool ok = true;
    for (int k = 0; ok && i0 + k < i1; ++k) {
        const int32_t u = a.list[i0 + k];
        const int32_t n = v.len[u] + a.fused;
        const int32_t Bu = v.budget[u];
        const int32_t tnew = v.next_pos[u] + a.fused - 1;
        const int32_t li = u / per_layer - a.layer0, b = (u / v.hkv) % v.batch, g = u % v.hkv;
        const bool need_victim = n > Bu;
        const int32_t nt = ceil_div(n, kDecTR);
        const int32_t sn = n - 1;   // fused: the new token's slot
        const int qb = k & 1;
        const uint8_t* nrow = smem + Lay::NROW + (warp * 2 + qb) * 2 * RB;
        float* imp = v.imp + (int64_t)u * v.cap;
        int32_t* pos = v.pos + (int64_t)u * v.cap;
        if (n > NCAP) {   // the host routes only units of at most NCAP tokens here
            if (lane == 0) atomicOr(v.err, DEVERR_STATE);
        }
        for (int j = lane * 32; j < n; j += 32 * 32) {   // the importance pass's lines, towards L2
            prefetch_global_l2(imp + j);
            prefetch_global_l2(pos + j);
        }
        if (!mbar_wait_bounded(&qfull[warp * 2 + qb], (uint32_t)(k >> 1) & 1u, v.err, kWaitQFull, (uint32_t)k)) {
            ok = false;
            break;
        }
        {
            const T* qraw = reinterpret_cast<const T*>(smem + Lay::QRAW + (warp * 2 + qb) * QB);
            for (int i = lane; i < G * D; i += 32) q_s[i] = Elem<T>::to_f(qraw[i]) * a.qscale;
        }
        __syncwarp();

        float2 qreg[G][QK_EPL / 2];
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < QK_EPL / 2; ++e)
                qreg[h][e] = *reinterpret_cast<const float2*>(q_s + h * D + qk_c * QK_EPL + 2 * e);
        float m_w[G];
        float m_own = -INFINITY, l_own = 0.f;
        float2 o2[G][EPL / 2];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            m_w[h] = -INFINITY;
#pragma unroll
            for (int e = 0; e < EPL / 2; ++e) o2[h][e] = make_float2(0.f, 0.f);
        }
        for (int32_t i = 0; i < nt; ++i, ++gj) {
            const int st = warp + kSmallWarps * (gj & 1);
            if (!mbar_wait_bounded(&full[st], (uint32_t)(gj >> 1) & 1u, v.err, kWaitFull, (uint32_t)(gj | (warp << 24)))) {
                ok = false;
                break;
            }
            const int32_t s0 = i * kDecTR;
            uint8_t* ktile = ring + st * 2 * TB;
            uint8_t* vtile = ktile + TB;
            const int32_t hi_r = min(kDecTR, n - s0);   // valid rows [0, hi_r)
            if (a.fused && sn >= s0 && sn < s0 + kDecTR) {
                // the new token's pool slot was loaded stale: patch the landed
                // tile from the staged rows, and write them to the pool
                const int r = sn - s0;
                const Raw nk = *reinterpret_cast<const Raw*>(nrow + lane * LB);
                const Raw nv = *reinterpret_cast<const Raw*>(nrow + RB + lane * LB);
                *reinterpret_cast<Raw*>(ktile + lin<RB>(r, pv_chunk) + pv_in) = nk;
                *reinterpret_cast<Raw*>(vtile + lin<RB>(r, pv_chunk) + pv_in) = nv;
                fence_proxy_async_smem();
                const int32_t pg = v.page_table[(int64_t)u * v.max_pages + (sn >> v.page_shift)];
                if (pg >= 0 && pg < v.pool_pages) {
                    uint8_t* kd = v.pool + (int64_t)pg * v.page_bytes + (int64_t)(sn & (v.page_tokens - 1)) * RB;
                    *reinterpret_cast<Raw*>(kd + lane * LB) = nk;
                    *reinterpret_cast<Raw*>(kd + (int64_t)v.page_tokens * RB + lane * LB) = nv;
                }
                __syncwarp();
            }
            // q.k: per sub-block, each lane's chunk of QK_SUB rows against q in
            // registers, then the partial sums reduce-scattered
            float sv[QK_NSUB];
#pragma unroll
            for (int sb = 0; sb < QK_NSUB; ++sb) {
                float part[QK_NV];
#pragma unroll
                for (int j = 0; j < QK_SUB; ++j) {
                    const int r = (sb * QK_SUB + j) * QK_RPW + qk_rg;
                    const uint4 raw = *reinterpret_cast<const uint4*>(ktile + lin<RB>(r, qk_c));
                    float x[QK_EPL];
                    Widen<T, QK_EPL>::run(raw, x);
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                        for (int e = 0; e < QK_EPL / 2; ++e)
                            acc = ffma2(make_float2(x[2 * e], x[2 * e + 1]), qreg[h][e], acc);
                        part[j * G + h] = acc.x + acc.y;
                    }
                }
                qk_reduce<QK_LPR / 2, QK_NV>(part, lane);
                const int r = (sb * QK_SUB + qk_step) * QK_RPW + qk_rg;
                sv[sb] = r < hi_r ? part[0] : -INFINITY;
            }
            bool big = false;
#pragma unroll
            for (int sb = 0; sb < QK_NSUB; ++sb) big |= sv[sb] > m_own + kDecLazy;
            if (__any_sync(0xffffffffu, big)) {
                float tmax = sv[0];
#pragma unroll
                for (int sb = 1; sb < QK_NSUB; ++sb) tmax = fmaxf(tmax, sv[sb]);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float mt = hk == h ? tmax : -INFINITY;
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
                    const float mn = fmaxf(m_w[h], mt);
                    const float scl = exp2f(m_w[h] - mn);
                    m_w[h] = mn;
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
                    ps[r * G + hk] = p;
                    if (rv && s0 + r < NCAP) S[(s0 + r) * G + hk] = sv[sb];
                }
            }
            __syncwarp();
            // p.v; a full tile has no per-row test, so its loads can be issued ahead
            auto pv_row = [&](int r) {
                const Raw raw = *reinterpret_cast<const Raw*>(vtile + lin<RB>(r, pv_chunk) + pv_in);
                float x[EPL];
                Widen<T, EPL>::run(raw, x);
                const float* pr = ps + r * G;
                float2 pp[G];
#pragma unroll
                for (int h = 0; h < G; ++h) pp[h] = make_float2(pr[h], pr[h]);
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int e = 0; e < EPL / 2; ++e)
                        o2[h][e] = ffma2(make_float2(x[2 * e], x[2 * e + 1]), pp[h], o2[h][e]);
            };
            if (hi_r == kDecTR) {
#pragma unroll
                for (int r = 0; r < kDecTR; ++r) pv_row(r);
            } else {
#pragma unroll
                for (int r = 0; r < kDecTR; ++r)
                    if (r < hi_r) pv_row(r);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
        }
        if (!ok) break;

        // the warp's state is the unit's: reference m_h, sum l_h over all rows
        float li_[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float t = (qk_own && hk == h) ? l_own : 0.f;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
            li_[h] = 1.0f / t;
        }
        {
            T* outp = reinterpret_cast<T*>(a.out) + (((int64_t)li * v.batch + b) * v.hq + (int64_t)g * G) * D;
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < EPL / 2; ++e) {
                    outp[h * D + lane * EPL + 2 * e] = Elem<T>::from_f(o2[h][e].x * li_[h]);
                    outp[h * D + lane * EPL + 2 * e + 1] = Elem<T>::from_f(o2[h][e].y * li_[h]);
                }
        }
        __syncwarp();   // S and the staged rows are read below

        // importance update + victim (smallest eligible (imp, -pos))
        unsigned long long kmin = ~0ull;
        int32_t smin = -1;
        float new_imp = -1.f;
        const int32_t lo = v.sink, hi = tnew - v.window;
        for (int32_t j = lane; j < n; j += 32) {
            const bool fresh = a.fused && j == sn;
            const float iv = fresh ? 0.f : imp[j];
            const int32_t pj = fresh ? tnew : pos[j];
            const float* srow = S + min(j, NCAP - 1) * G;   // j < NCAP for every unit routed here
            float inc = 0.f;
#pragma unroll
            for (int h = 0; h < G; ++h) inc += exp2f(srow[h] - m_w[h]) * li_[h];
            const bool grows = !v.recent_only || pj >= tnew - v.window;
            const float nw = grows ? iv + inc : iv;
            imp[j] = nw;
            if (fresh) {
                pos[j] = tnew;
                new_imp = nw;
            }
            if (need_victim && pj >= lo && pj <= hi) {
                const unsigned long long key =
                    ((unsigned long long)__float_as_uint(nw) << 32) | (unsigned long long)(~(uint32_t)pj);
                if (key < kmin) {
                    kmin = key;
                    smin = j;
                }
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const unsigned long long ok2 = __shfl_xor_sync(0xffffffffu, kmin, o);
            const int32_t os = __shfl_xor_sync(0xffffffffu, smin, o);
            if (ok2 < kmin) {
                kmin = ok2;
                smin = os;
            }
            new_imp = fmaxf(new_imp, __shfl_xor_sync(0xffffffffu, new_imp, o));
        }
        const int32_t vs = need_victim ? smin : -1;
        if (!a.fused) {
            if (lane == 0) v.victim[u] = vs;
        } else {
            const bool cut = a.evict && vs >= 0;
            if (lane == 0) {
                v.victim[u] = cut ? -1 : vs;
                v.len[u] = cut ? n - 1 : n;
                v.next_pos[u] = tnew + 1;
            }
            if (cut && vs != sn) {
                // the new token (last slot) moves into the victim's slot
                const int32_t pd = v.page_table[(int64_t)u * v.max_pages + (vs >> v.page_shift)];
                if (pd >= 0 && pd < v.pool_pages) {
                    uint8_t* kd = v.pool + (int64_t)pd * v.page_bytes + (int64_t)(vs & (v.page_tokens - 1)) * RB;
                    *reinterpret_cast<Raw*>(kd + lane * LB) = *reinterpret_cast<const Raw*>(nrow + lane * LB);
                    *reinterpret_cast<Raw*>(kd + (int64_t)v.page_tokens * RB + lane * LB) =
                        *reinterpret_cast<const Raw*>(nrow + RB + lane * LB);
                } else if (lane == 0) {
                    atomicOr(v.err, DEVERR_PAGE);
                }
                if (lane == 0) {
                    imp[vs] = new_imp;
                    pos[vs] = tnew;
                }
            }
            if (v.debug && cut) {
                __syncwarp();
                poison_slot(v, u, sn, lane, 32);   // the last slot is vacated
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&qempty[warp * 2 + qb]);   // q, staged rows and S are free
    }
    __syncwarp();
    __syncthreads();
}

template <typename T, int D, int G>
cudaError_t decode_small_launch_one(const SmallArgs& a, const CUtensorMap& tmap, int n_ctas, cudaStream_t s) {
    constexpr int smem = SmallLayout<T, D, G>::TOTAL;
    const cudaError_t e = func_smem_optin(reinterpret_cast<const void*>(k_decode_small<T, D, G>), smem);
    if (e != cudaSuccess) return e;
    k_decode_small<T, D, G><<<n_ctas, kSmallThreads, smem, s>>>(a, tmap);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t decode_small_launch_g(const SmallArgs& a, const CUtensorMap& tmap, int group, int n_ctas, cudaStream_t s) {
    switch (group) {
        case 1: return decode_small_launch_one<T, D, 1>(a, tmap, n_ctas, s);
        case 2: return decode_small_launch_one<T, D, 2>(a, tmap, n_ctas, s);
        case 4: return decode_small_launch_one<T, D, 4>(a, tmap, n_ctas, s);
        case 8: return decode_small_launch_one<T, D, 8>(a, tmap, n_ctas, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace hikv
