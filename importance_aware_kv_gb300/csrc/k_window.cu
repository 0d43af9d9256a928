// Prefill importance from an observation window of queries (setup step).
//
// The importance of each prompt token starts as its attention column summed
// over the last nq prompt queries and the G query heads of its group, with
// causal masking (HiKV sec. III-D initialises importance from prefill
// attention summed over a window of late queries; SnapKV's observation
// window, blog sec. 3).  Queries are applied in position order so each
// token's running fp32 score follows the same per-query accumulation as a
// decode step.
//
// Two passes over the unit's keys, split into chunks of kWinChunk tokens:
//   pass 1  per chunk and query: running max and sum of 2^(s'-m) over the
//           tokens the query may see -> partials (m, l) in a scratch buffer;
//   pass 2  merge the partials of the unit, recompute the logits and add
//           sum_h 2^(s'-m) / l per query, in query order, to each token.
// This is a small dense contraction ([nq*G, d] x [d, n]) done once per
// prompt; it runs on CUDA cores, it is not part of the timed decode step.
#include "hikv_internal.cuh"

namespace hikv {
namespace {

constexpr int kWinThreads = 256;
constexpr int kWinTT = 32;   // tokens per sub-tile
constexpr int kWinQB = 64;   // query vectors per block

template <typename T>
__device__ void load_k_tile(const View& v, int32_t u, int32_t s0, int32_t n, int d, float* Ks) {
    // Ks [kWinTT][d] fp32; rows past n are zero
    for (int i = threadIdx.x; i < kWinTT * d; i += kWinThreads) {
        const int r = i / d, c = i % d;
        const int32_t s = s0 + r;
        float x = 0.f;
        if (s < n) {
            const uint8_t* p = row_ptr(v, u, s, false);
            if (p) x = Elem<T>::to_f(reinterpret_cast<const T*>(p)[c]);
        }
        Ks[r * (d + 1) + c] = x;
    }
}

// S[t][q] for the kWinTT tokens of Ks and query vectors [qb, qb+kWinQB) of Qs.
__device__ void tile_logits(const float* Ks, const float* Qs, int d, int qb, int nqv, float* St) {
    const int tq = threadIdx.x % 16, tt = threadIdx.x / 16;   // 16 x 16 threads
    float acc[2][4] = {};
    const int q0 = qb + tq * 4;
    for (int c = 0; c < d; ++c) {
        const float k0 = Ks[(tt * 2) * (d + 1) + c];
        const float k1 = Ks[(tt * 2 + 1) * (d + 1) + c];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int q = q0 + j;
            const float qv = q < nqv ? Qs[q * (d + 1) + c] : 0.f;
            acc[0][j] = fmaf(k0, qv, acc[0][j]);
            acc[1][j] = fmaf(k1, qv, acc[1][j]);
        }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int j = 0; j < 4; ++j) St[(tt * 2 + r) * kWinQB + tq * 4 + j] = acc[r][j];
}

template <typename T>
__device__ void load_queries(const WindowArgs& a, int32_t u, float* Qs) {
    const View& v = a.v;
    const int d = v.d, G = v.group, nq = a.nq;
    const int32_t per_layer = v.batch * v.hkv;
    const int32_t li = u / per_layer - a.layer0;
    const int32_t b = (u / v.hkv) % v.batch, g = u % v.hkv;
    // query vector qv = hh * nq + i  <->  q[li][b][g*G+hh][i][:]
    const T* base = reinterpret_cast<const T*>(a.q) +
                    (((int64_t)li * v.batch + b) * v.hq + (int64_t)g * G) * nq * d;
    for (int i = threadIdx.x; i < G * nq * d; i += kWinThreads) {
        const int qv = i / d, c = i % d;
        Qs[qv * (d + 1) + c] = Elem<T>::to_f(base[(int64_t)qv * d + c]) * a.qscale;
    }
}

template <typename T>
__global__ void __launch_bounds__(kWinThreads) k_window_p1(WindowArgs a) {
    extern __shared__ float wsm[];
    const View& v = a.v;
    const int d = v.d;
    const int32_t u = a.u0 + blockIdx.y;
    const int32_t n = v.len[u];
    const int32_t c0 = blockIdx.x * a.chunk;
    const int nqv = v.group * a.nq;
    float* part = a.part + (((int64_t)u * a.nchunks_max + blockIdx.x) * nqv) * 2;
    if (c0 >= n) {
        for (int q = threadIdx.x; q < nqv; q += kWinThreads) {
            part[2 * q] = -INFINITY;
            part[2 * q + 1] = 0.f;
        }
        return;
    }
    const int32_t c1 = min(n, c0 + a.chunk);
    const int32_t tnew = v.next_pos[u] - 1;
    float* Qs = wsm;                          // [nqv][d+1]
    float* Ks = Qs + nqv * (d + 1);           // [TT][d+1]
    float* St = Ks + kWinTT * (d + 1);        // [TT][QB]
    int32_t* Ps = reinterpret_cast<int32_t*>(St + kWinTT * kWinQB);  // [TT]
    load_queries<T>(a, u, Qs);
    // running (m, l) per query vector
    float* ML = reinterpret_cast<float*>(Ps + kWinTT);  // [nqv][2]
    for (int q = threadIdx.x; q < nqv; q += kWinThreads) {
        ML[2 * q] = -INFINITY;
        ML[2 * q + 1] = 0.f;
    }
    for (int32_t s0 = c0; s0 < c1; s0 += kWinTT) {
        __syncthreads();
        load_k_tile<T>(v, u, s0, c1, d, Ks);
        for (int r = threadIdx.x; r < kWinTT; r += kWinThreads)
            Ps[r] = (s0 + r < c1) ? v.pos[(int64_t)u * v.cap + s0 + r] : INT32_MAX;
        __syncthreads();
        for (int qb = 0; qb < nqv; qb += kWinQB) {
            tile_logits(Ks, Qs, d, qb, nqv, St);
            __syncthreads();
            const int q = qb + threadIdx.x;
            if (threadIdx.x < kWinQB && q < nqv) {
                const int i = q % a.nq;                 // query index within the window
                const int32_t qpos = tnew - a.nq + 1 + i;
                float m = ML[2 * q], l = ML[2 * q + 1];
                float tm = -INFINITY;
                for (int r = 0; r < kWinTT; ++r)
                    if (Ps[r] <= qpos) tm = fmaxf(tm, St[r * kWinQB + threadIdx.x]);
                if (tm > -INFINITY) {
                    const float nm = fmaxf(m, tm);
                    float acc = (l > 0.f) ? l * exp2f(m - nm) : 0.f;
                    for (int r = 0; r < kWinTT; ++r)
                        if (Ps[r] <= qpos) acc += exp2f(St[r * kWinQB + threadIdx.x] - nm);
                    ML[2 * q] = nm;
                    ML[2 * q + 1] = acc;
                }
            }
            __syncthreads();
        }
    }
    __syncthreads();
    for (int q = threadIdx.x; q < nqv; q += kWinThreads) {
        part[2 * q] = ML[2 * q];
        part[2 * q + 1] = ML[2 * q + 1];
    }
}

template <typename T>
__global__ void __launch_bounds__(kWinThreads) k_window_p2(WindowArgs a) {
    extern __shared__ float wsm[];
    const View& v = a.v;
    const int d = v.d, G = v.group, nq = a.nq;
    const int32_t u = a.u0 + blockIdx.y;
    const int32_t n = v.len[u];
    const int32_t c0 = blockIdx.x * a.chunk;
    if (c0 >= n) return;
    const int32_t c1 = min(n, c0 + a.chunk);
    const int32_t tnew = v.next_pos[u] - 1;
    const int nqv = G * nq;
    const int nch = ceil_div(n, a.chunk);
    float* Qs = wsm;
    float* Ks = Qs + nqv * (d + 1);
    float* St = Ks + kWinTT * (d + 1);
    int32_t* Ps = reinterpret_cast<int32_t*>(St + kWinTT * kWinQB);
    float* MF = reinterpret_cast<float*>(Ps + kWinTT);   // [nqv] final max
    float* LI = MF + nqv;                                 // [nqv] 1 / l
    float* Pt = LI + nqv;                                 // [TT][nqv] probabilities
    load_queries<T>(a, u, Qs);
    const float* part = a.part + ((int64_t)u * a.nchunks_max) * nqv * 2;
    for (int q = threadIdx.x; q < nqv; q += kWinThreads) {
        float m = -INFINITY;
        for (int cc = 0; cc < nch; ++cc) m = fmaxf(m, part[((int64_t)cc * nqv + q) * 2]);
        float l = 0.f;
        for (int cc = 0; cc < nch; ++cc) {
            const float lc = part[((int64_t)cc * nqv + q) * 2 + 1];
            if (lc > 0.f) l += lc * exp2f(part[((int64_t)cc * nqv + q) * 2] - m);
        }
        MF[q] = m;
        LI[q] = 1.0f / l;
    }
    for (int32_t s0 = c0; s0 < c1; s0 += kWinTT) {
        __syncthreads();
        load_k_tile<T>(v, u, s0, c1, d, Ks);
        for (int r = threadIdx.x; r < kWinTT; r += kWinThreads)
            Ps[r] = (s0 + r < c1) ? v.pos[(int64_t)u * v.cap + s0 + r] : INT32_MAX;
        __syncthreads();
        for (int qb = 0; qb < nqv; qb += kWinQB) {
            tile_logits(Ks, Qs, d, qb, nqv, St);
            __syncthreads();
            for (int i = threadIdx.x; i < kWinTT * kWinQB; i += kWinThreads) {
                const int r = i / kWinQB, qq = i % kWinQB, q = qb + qq;
                if (q >= nqv) continue;
                const int32_t qpos = tnew - nq + 1 + q % nq;
                Pt[r * nqv + q] = (Ps[r] <= qpos) ? exp2f(St[r * kWinQB + qq] - MF[q]) * LI[q] : 0.f;
            }
            __syncthreads();
        }
        // per token: queries in position order, heads ascending within a query
        for (int r = threadIdx.x; r < kWinTT; r += kWinThreads) {
            const int32_t s = s0 + r;
            if (s >= c1) continue;
            const int64_t mi = (int64_t)u * v.cap + s;
            float imp = v.imp[mi];
            for (int i = 0; i < nq; ++i) {
                float inc = 0.f;
                for (int hh = 0; hh < G; ++hh) inc += Pt[r * nqv + hh * nq + i];
                imp = imp + inc;
            }
            v.imp[mi] = imp;
        }
    }
}

size_t window_smem(int d, int nqv) {
    size_t f = (size_t)nqv * (d + 1) + (size_t)kWinTT * (d + 1) + (size_t)kWinTT * kWinQB;
    f += kWinTT;                       // Ps
    f += 2 * (size_t)nqv;              // ML or MF+LI
    f += (size_t)kWinTT * nqv;         // Pt (pass 2)
    return f * 4;
}

}  // namespace

size_t window_smem_bytes(int d, int nqv) { return window_smem(d, nqv); }

cudaError_t launch_window(const WindowArgs& a, int dtype, int d, int group, cudaStream_t s) {
    const int nqv = group * a.nq;
    const size_t smem = window_smem(d, nqv);
    dim3 grid(a.nchunks_grid, a.nunits);
    cudaError_t e;
    if (dtype == 0) {
        e = func_smem_optin(reinterpret_cast<const void*>(k_window_p1<float>), smem);
        if (e == cudaSuccess) e = func_smem_optin(reinterpret_cast<const void*>(k_window_p2<float>), smem);
        if (e != cudaSuccess) return e;
        k_window_p1<float><<<grid, kWinThreads, smem, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        k_window_p2<float><<<grid, kWinThreads, smem, s>>>(a);
    } else {
        e = func_smem_optin(reinterpret_cast<const void*>(k_window_p1<__nv_bfloat16>), smem);
        if (e == cudaSuccess) e = func_smem_optin(reinterpret_cast<const void*>(k_window_p2<__nv_bfloat16>), smem);
        if (e != cudaSuccess) return e;
        k_window_p1<__nv_bfloat16><<<grid, kWinThreads, smem, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        k_window_p2<__nv_bfloat16><<<grid, kWinThreads, smem, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace hikv
