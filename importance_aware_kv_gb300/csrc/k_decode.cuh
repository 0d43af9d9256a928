// Fused decode attention + importance update + victim argmin.
//
// One thread-block cluster per unit (layer, batch, KV head); its CS CTAs split
// the unit's n live slots into equal chunks.  Per CTA:
//   producer warp  streams the chunk in 16-row tiles, each tile's K rows and
//                  V rows together, HBM -> shared memory with 1-D TMA bulk
//                  copies into an NSTAGE ring (mbarrier full/empty pairs,
//                  bounded waits);
//   4 consumer warps, each owning every 4th row of a tile, keep a private
//   online softmax (running max m_w, sum l_w, unnormalised O_w):
//     logits s'_hj = <q_h * scale * log2 e, k_j> for the G query heads of the
//     group -- a lane holds d/32 elements of a row, a warp reduce-scatter
//     leaves one (row, head) sum per lane; logits are kept (shared memory, or
//     an L2-resident global buffer for very long chunks) for the importance
//     update; then p = 2^(s' - m_w), O_w += p v_j for the same tile's V rows.
//   CTA merge of the 4 warp states, then a cluster merge by remote stores
//   into shared memory (DSMEM) before one cluster barrier:
//     m = max_c m_c, l = sum_c l_c 2^(m_c - m); out_h = sum_c O_c[h] 2^(m_c - m) / l;
//     importance imp_j += sum_h 2^(s'_hj - m_h) / l_h (fp32 add, heads
//     ascending), and the eligible slot with the smallest (imp, -pos) is the
//     step's victim, gathered in CTA 0 by a second remote store + barrier.
//
// Method: decode attention P = softmax(q K^T), O = P V (HiKV sec. II-A; Kelle
// summary sec. 2.2); importance accumulates P summed over the group's heads
// (blog sec. 3 "H2O", sec. 5.2); the victim is the least important token that
// is neither a sink nor in the recent window, ties evicting the higher
// position (blog sec. 3 "H2O"/"StreamingLLM").  The argmin stands in for the
// min-search that Kelle's systolic evictor runs alongside attention (Kelle
// summary sec. 5.3) and HiKV's min-heap (sec. III-B).
#pragma once

#include "hikv_internal.cuh"

namespace hikv {

constexpr int kDecNCW = 4;                       // consumer warps
constexpr int kDecThreads = (kDecNCW + 1) * 32;  // + producer warp
constexpr int kDecTR = 16;                       // rows per tile
constexpr int kDecStages = 4;

// reduce-scatter of N0 per-lane values over the warp.  Stage k exchanges half
// of the remaining values with the lane 16 >> k away; afterwards lane l holds
// the sum over 32 / N0 lanes of value index l / (32 / N0), and the butterfly
// in warp_reduce_scatter_full completes it to the full warp sum.
template <int N, int N0>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[N], int lane) {
    if constexpr (N == 1) {
        return v[0];
    } else {
        constexpr int H = N / 2;
        constexpr int off = 16 * N / N0;
        const bool upper = (lane & off) != 0;
        float nv[H];
#pragma unroll
        for (int i = 0; i < H; ++i) {
            float send = upper ? v[i] : v[i + H];
            float keep = upper ? v[i + H] : v[i];
            nv[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
        return warp_reduce_scatter<H, N0>(nv, lane);
    }
}

template <int N>
__device__ __forceinline__ float warp_reduce_scatter_full(float (&v)[N], int lane) {
    float r = warp_reduce_scatter<N, N>(v, lane);
#pragma unroll
    for (int o = 16 / N; o >= 1; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    return r;
}

struct DecSmem {
    // byte offsets into dynamic shared memory
    uint32_t ring, bars, ws, recv, small, S, simp, spos, total;
};

template <typename T, int D, int G>
__host__ __device__ constexpr uint32_t dec_ring_bytes() {
    return (uint32_t)kDecStages * 2 * kDecTR * D * sizeof(T);
}

template <typename T, int D, int G>
__host__ __device__ inline DecSmem dec_layout(bool smem_s, int chunk_cap) {
    DecSmem L{};
    uint32_t off = 0;
    L.ring = off;                                 // also the warp-partial O buffer after streaming
    off += dec_ring_bytes<T, D, G>();
    L.bars = off;
    off += 2 * kDecStages * 8;
    L.ws = off;                                   // [NCW][2][32] per-warp broadcast scratch
    off += kDecNCW * 2 * 32 * 4;
    L.recv = off;                                 // O slices from every CTA: G*D + kMaxCS floats
    off += (G * D + kMaxCS) * 4;
    L.small = off;
    off += 4096;
    L.S = off;
    if (smem_s) {
        off += (uint32_t)chunk_cap * G * 4;
        off = (off + 15) & ~15u;
        L.simp = off;
        off += (uint32_t)chunk_cap * 4;
        L.spos = off;
        off += (uint32_t)chunk_cap * 4;
    } else {
        L.simp = L.spos = off;
    }
    L.total = (off + 127) & ~127u;
    return L;
}

template <typename T, int D, int G, bool SMEM_S>
__global__ void __launch_bounds__(kDecThreads, (G <= 4 ? 4 : 2)) k_decode(const DecodeArgs a) {
    constexpr int RB = D * (int)sizeof(T);   // row bytes
    constexpr int TB = kDecTR * RB;          // tile bytes (K or V)
    constexpr int EPL = D / 32;              // elements per lane
    constexpr int LB = EPL * (int)sizeof(T); // bytes per lane
    constexpr int RPW = kDecTR / kDecNCW;    // rows per warp per tile
    constexpr int NV = RPW * G;              // logits per warp per tile
    constexpr int NCT = kDecNCW * 32;        // consumer threads
    static_assert(NV <= 32 && (NV & (NV - 1)) == 0, "group size");
    using Raw = typename RawVec<LB>::type;

    extern __shared__ __align__(128) uint8_t smem[];
    const View& v = a.v;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    const DecSmem L = dec_layout<T, D, G>(SMEM_S, a.chunk_cap);
    uint8_t* ring = smem + L.ring;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* empty = full + kDecStages;
    float* ws = reinterpret_cast<float*>(smem + L.ws);        // [NCW][2][32]
    float* orecv = reinterpret_cast<float*>(smem + L.recv);   // [CS][per]
    float* sm = reinterpret_cast<float*>(smem + L.small);
    float* m_recv = sm;                        // [kMaxCS][G]  (128)
    float* l_recv = sm + 128;                  // [kMaxCS][G]  (128)
    float* beta = sm + 256;                    // [kMaxCS][G]  (128)
    float* mw_s = sm + 384;                    // [NCW][G]     (32)
    float* lw_s = sm + 416;                    // [NCW][G]     (32)
    float* wsc = sm + 448;                     // [NCW][G]     (32)
    float* m_c = sm + 480;                     // [G]
    float* l_c = sm + 488;                     // [G]
    float* mfin = sm + 496;                    // [G]
    float* linv = sm + 504;                    // [G]
    unsigned long long* akey = reinterpret_cast<unsigned long long*>(sm + 512);  // [kMaxCS]
    int32_t* aslot = reinterpret_cast<int32_t*>(akey + kMaxCS);                  // [kMaxCS]
    unsigned long long* wkey = reinterpret_cast<unsigned long long*>(aslot + kMaxCS);  // [NCW]
    int32_t* wslot = reinterpret_cast<int32_t*>(wkey + kDecNCW);                     // [NCW]
    volatile int32_t* abort_flag = wslot + kDecNCW;
    float* S_smem = reinterpret_cast<float*>(smem + L.S);
    float* simp = reinterpret_cast<float*>(smem + L.simp);
    int32_t* spos = reinterpret_cast<int32_t*>(smem + L.spos);

    const int32_t c = (int32_t)cluster_ctarank();
    const int32_t CS = (int32_t)cluster_nctarank();
    const int32_t u = a.order[blockIdx.y];
    const int32_t per_layer = v.batch * v.hkv;
    const int32_t li = u / per_layer - a.layer0;
    const int32_t b = (u / v.hkv) % v.batch;
    const int32_t g = u % v.hkv;
    const int32_t n = v.len[u];
    const int32_t Bu = v.budget[u];
    const int32_t tnew = v.next_pos[u] - 1;
    const bool need_victim = n > Bu;
    const int32_t chunk = ceil_div(n, CS);
    const int32_t t0 = min(n, c * chunk);
    int32_t t1 = min(n, t0 + chunk);
    int32_t cnt = t1 - t0;
    if (SMEM_S && cnt > a.chunk_cap) {   // host sizes chunk_cap; never taken
        if (threadIdx.x == 0) atomicOr(v.err, DEVERR_STATE);
        cnt = a.chunk_cap;
        t1 = t0 + cnt;
    }
    const int32_t first_blk = t0 / kDecTR;
    const int32_t nt = cnt > 0 ? (t1 - 1) / kDecTR - first_blk + 1 : 0;
    const int64_t qbase = (((int64_t)li * v.batch + b) * v.hq + (int64_t)g * G) * D;
    const int32_t per = ceil_div(G * D, CS);   // output elements finalised per CTA

    float* Sb = SMEM_S ? S_smem : a.logits + ((int64_t)u * v.cap) * G;
    const int32_t s_off = SMEM_S ? t0 : 0;   // S index of slot s = (s - s_off) * G

    if (tid == 0) {
        for (int s = 0; s < kDecStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kDecNCW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kDecNCW) {
        // ---------------- producer ----------------
        if (lane == 0) {
            int it = 0;
            for (; it < nt; ++it) {
                if (*abort_flag) break;
                const int st = it % kDecStages;
                const uint32_t round = (uint32_t)(it / kDecStages);
                if (!mbar_wait_bounded(&empty[st], (round & 1u) ^ 1u, v.err)) {
                    *abort_flag = 1;
                    break;
                }
                const int32_t s0 = max(t0, (first_blk + it) * kDecTR);
                const int32_t s1 = min(t1, (first_blk + it + 1) * kDecTR);
                const uint8_t* ksrc = row_ptr(v, u, s0, false);
                const uint8_t* vsrc = row_ptr(v, u, s0, true);
                const uint32_t bytes = (uint32_t)(s1 - s0) * RB;
                if (ksrc == nullptr || vsrc == nullptr) {
                    // unmapped page: complete the stage without data
                    *abort_flag = 1;
                    mbar_arrive(&full[st]);
                    break;
                }
                mbar_arrive_expect_tx(&full[st], 2 * bytes);
                bulk_g2s(ring + st * 2 * TB, ksrc, bytes, &full[st]);
                bulk_g2s(ring + st * 2 * TB + TB, vsrc, bytes, &full[st]);
            }
            if (*abort_flag) {
                // let copies already in flight land before the CTA can exit
                for (int k = max(0, it - kDecStages); k < it; ++k)
                    mbar_wait_bounded(&full[k % kDecStages], (uint32_t)(k / kDecStages) & 1u, v.err);
            }
        }
        __syncwarp();
        cluster_sync_all();
        cluster_sync_all();
        return;
    }

    // ---------------- consumers ----------------
    const int ctid = tid;  // 0..127
    float qr[G][EPL];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const Raw raw = *reinterpret_cast<const Raw*>(reinterpret_cast<const T*>(a.q) + qbase +
                                                      (int64_t)h * D + lane * EPL);
        Widen<T, EPL>::run(raw, qr[h]);
#pragma unroll
        for (int e = 0; e < EPL; ++e) qr[h][e] *= a.qscale;
    }
    if (SMEM_S) {
        for (int j = ctid; j < cnt; j += NCT) {
            simp[j] = v.imp[(int64_t)u * v.cap + t0 + j];
            spos[j] = v.pos[(int64_t)u * v.cap + t0 + j];
        }
    }

    float* ws_s = ws + warp * 64;        // this warp's logits of the tile, [k*G + h]
    float* ws_p = ws_s + 32;             // this warp's probabilities of the tile
    float m_w[G], l_w[G], o[G][EPL];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m_w[h] = -INFINITY;
        l_w[h] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[h][e] = 0.f;
    }
    constexpr int stride = 32 / NV;
    const int vi = lane / stride;             // (row, head) value this lane ends up with
    const int vk = vi / G, vh = vi % G;
    const bool writer = (lane & (stride - 1)) == 0;

    for (int i = 0; i < nt; ++i) {
        if (*abort_flag) break;
        const int st = i % kDecStages;
        if (!mbar_wait_bounded(&full[st], (uint32_t)(i / kDecStages) & 1u, v.err)) {
            *abort_flag = 1;
            break;
        }
        const int32_t s0 = max(t0, (first_blk + i) * kDecTR);
        const int32_t rows = min(t1, (first_blk + i + 1) * kDecTR) - s0;
        const uint8_t* ktile = ring + st * 2 * TB;
        const uint8_t* vtile = ktile + TB;
        // logits of this warp's rows
        float acc[NV];
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
            const int r = warp + kDecNCW * k;
            float x[EPL];
            if (r < rows) {
                Raw raw = *reinterpret_cast<const Raw*>(ktile + r * RB + lane * LB);
                Widen<T, EPL>::run(raw, x);
            } else {
#pragma unroll
                for (int e = 0; e < EPL; ++e) x[e] = 0.f;
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float sacc = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) sacc = fmaf(x[e], qr[h][e], sacc);
                acc[k * G + h] = sacc;
            }
        }
        const float val = warp_reduce_scatter_full<NV>(acc, lane);
        const int vr = warp + kDecNCW * vk;       // tile row of this lane's value
        if (writer) {
            ws_s[vi] = (vr < rows) ? val : -INFINITY;
            if (vr < rows) Sb[(int64_t)(s0 + vr - s_off) * G + vh] = val;
        }
        __syncwarp();
        // tile max per head over this warp's valid rows; new running max
        float m_new[G], scl[G];
        bool rescale = false;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float tm = -INFINITY;
#pragma unroll
            for (int k = 0; k < RPW; ++k) tm = fmaxf(tm, ws_s[k * G + h]);
            m_new[h] = fmaxf(m_w[h], tm);
            scl[h] = (m_new[h] == m_w[h]) ? 1.f : exp2f(m_w[h] - m_new[h]);   // m_w = -inf -> 0
            rescale |= (m_new[h] != m_w[h]);
        }
        if (writer) {
            float mh = m_new[0];
#pragma unroll
            for (int h = 1; h < G; ++h)
                if (vh == h) mh = m_new[h];
            ws_p[vi] = (vr < rows) ? exp2f(val - mh) : 0.f;
        }
        __syncwarp();
        if (rescale) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                l_w[h] *= scl[h];
#pragma unroll
                for (int e = 0; e < EPL; ++e) o[h][e] *= scl[h];
            }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) m_w[h] = m_new[h];
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
            const int r = warp + kDecNCW * k;
            if (r < rows) {
                float p[G];
#pragma unroll
                for (int h = 0; h < G; ++h) p[h] = ws_p[k * G + h];
                Raw raw = *reinterpret_cast<const Raw*>(vtile + r * RB + lane * LB);
                float x[EPL];
                Widen<T, EPL>::run(raw, x);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    l_w[h] += p[h];
#pragma unroll
                    for (int e = 0; e < EPL; ++e) o[h][e] = fmaf(p[h], x[e], o[h][e]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }

    // ---- CTA merge of the 4 warp states (ring reused for the O partials) ----
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            mw_s[warp * G + h] = m_w[h];
            lw_s[warp * G + h] = l_w[h];
        }
    }
    named_bar_sync(1, NCT);   // every warp is done with the ring
    float* red = reinterpret_cast<float*>(ring);   // [NCW][G][D]
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < EPL; ++e) red[(warp * G + h) * D + lane * EPL + e] = o[h][e];
    if (ctid < G) {
        float m = -INFINITY;
        for (int w = 0; w < kDecNCW; ++w) m = fmaxf(m, mw_s[w * G + ctid]);
        float l = 0.f;
        for (int w = 0; w < kDecNCW; ++w) {
            const float mw = mw_s[w * G + ctid];
            const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - m);
            wsc[w * G + ctid] = f;
            l += lw_s[w * G + ctid] * f;
        }
        m_c[ctid] = m;
        l_c[ctid] = l;
    }
    named_bar_sync(1, NCT);
    // push (m_c, l_c) to every CTA of the cluster and O_c slices to their owners
    if (ctid < CS * G) {
        const int cc = ctid / G, h = ctid % G;
        dsmem_st_f32(dsmem_addr(&m_recv[c * G + h], (uint32_t)cc), m_c[h]);
        dsmem_st_f32(dsmem_addr(&l_recv[c * G + h], (uint32_t)cc), l_c[h]);
    }
    for (int idx = ctid; idx < G * D; idx += NCT) {
        const int h = idx / D;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kDecNCW; ++w) s += red[w * G * D + idx] * wsc[w * G + h];
        const int owner = idx / per, loc = idx - owner * per;
        dsmem_st_f32(dsmem_addr(&orecv[c * per + loc], (uint32_t)owner), s);
    }

    __syncwarp();
    cluster_sync_all();  // #1: every CTA's (m_c, l_c) and O slices are in place

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
            const int idx = c * per + loc;
            if (idx >= G * D) break;
            const int h = idx / D;
            float s = 0.f;
            for (int cc = 0; cc < CS; ++cc) s += orecv[cc * per + loc] * beta[cc * G + h];
            outp[idx] = Elem<T>::from_f(s);
        }
    }
    // importance update + local victim
    {
        float mf[G], li_[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            mf[h] = mfin[h];
            li_[h] = linv[h];
        }
        unsigned long long kmin = ~0ull;
        int32_t smin = -1;
        const int32_t lo = v.sink, hi = tnew - v.window;
        for (int j = ctid; j < cnt; j += NCT) {
            const int32_t slot = t0 + j;
            const float* srow = Sb + (int64_t)(slot - s_off) * G;
            float inc = 0.f;
#pragma unroll
            for (int h = 0; h < G; ++h) inc += exp2f(srow[h] - mf[h]) * li_[h];
            const int64_t mi = (int64_t)u * v.cap + slot;
            const float old = SMEM_S ? simp[j] : v.imp[mi];
            const float nw = old + inc;
            v.imp[mi] = nw;
            if (need_victim) {
                const int32_t p = SMEM_S ? spos[j] : v.pos[mi];
                if (p >= lo && p <= hi) {
                    const unsigned long long key =
                        ((unsigned long long)__float_as_uint(nw) << 32) | (unsigned long long)(~(uint32_t)p);
                    if (key < kmin) {
                        kmin = key;
                        smin = slot;
                    }
                }
            }
        }
        if (need_victim) {
#pragma unroll
            for (int o2 = 16; o2 >= 1; o2 >>= 1) {
                const unsigned long long ok = __shfl_xor_sync(0xffffffffu, kmin, o2);
                const int32_t os = __shfl_xor_sync(0xffffffffu, smin, o2);
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
    }
    named_bar_sync(1, NCT);
    if (ctid == 0 && need_victim) {
        unsigned long long k = ~0ull;
        int32_t s = -1;
        for (int w = 0; w < kDecNCW; ++w)
            if (wkey[w] < k) {
                k = wkey[w];
                s = wslot[w];
            }
        dsmem_st_u64(dsmem_addr(&akey[c], 0u), k);
        dsmem_st_s32(dsmem_addr(&aslot[c], 0u), s);
    }

    __syncwarp();
    cluster_sync_all();  // #2: every CTA's local victim is in CTA 0

    if (c == 0 && ctid == 0) {
        int32_t vs = -1;
        if (need_victim) {
            unsigned long long k = ~0ull;
            for (int cc = 0; cc < CS; ++cc)
                if (akey[cc] < k) {
                    k = akey[cc];
                    vs = aslot[cc];
                }
        }
        v.victim[u] = vs;
    }
}

}  // namespace hikv

namespace hikv {

template <typename T, int D, int G, bool SM>
cudaError_t decode_launch_one(const DecodeArgs& a, size_t smem, cudaStream_t s) {
    auto kern = k_decode<T, D, G, SM>;
    static size_t smem_set = 0;  // largest dynamic smem opted into so far
    if (smem > smem_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        smem_set = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.cs, (unsigned)a.n_units, 1);
    cfg.blockDim = dim3(kDecThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)a.cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename T, int D, bool SM>
cudaError_t decode_launch_g(const DecodeArgs& a, int group, size_t smem, cudaStream_t s) {
    switch (group) {
        case 1: return decode_launch_one<T, D, 1, SM>(a, smem, s);
        case 2: return decode_launch_one<T, D, 2, SM>(a, smem, s);
        case 4: return decode_launch_one<T, D, 4, SM>(a, smem, s);
        case 8: return decode_launch_one<T, D, 8, SM>(a, smem, s);
        default: return cudaErrorInvalidValue;
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
    cudaError_t decode_launch_##NAME(const DecodeArgs& a, int group, bool smem_path, size_t smem,   \
                                     cudaStream_t s) {                                              \
        return smem_path ? decode_launch_g<T, D, true>(a, group, smem, s)                           \
                         : decode_launch_g<T, D, false>(a, group, smem, s);                         \
    }                                                                                               \
    size_t decode_smem_##NAME(int group, bool smem_path, int chunk_cap) {                           \
        return decode_smem_t<T, D>(group, smem_path, chunk_cap);                                    \
    }                                                                                               \
    }
