// HiKV prefill initialisation: banded attention-column scores.
//
// HiKV (sec. III-D) initialises its dual bank from the prefill attention:
// every prompt token l gets IS(l) = sum_{k=0}^{band-1} P_{l+k}[l] -- the IS
// definition of sec. III-B with band = B_I / 2 -- the attention its column
// receives from the band of queries that starts at its own position, causally
// masked (queries past the prompt do not exist and add nothing).  Under GQA
// the G query heads of a KV group add into one score per KV head.
//
// Two passes per layer, fp32 CUDA-core arithmetic on both dtypes:
//   k_band_stats   per (unit, tile of 64 query rows; a row is a (position,
//                  head) pair): the causal softmax statistics of every row
//                  over the keys at positions <= its own -- per-thread online
//                  maxima and sums over the columns a thread owns, merged
//                  across the row's 16 threads at the end;
//   k_band_scores  per (unit, tile of 64 keys): the probabilities
//                  2^(s'_ij - m_i) / l_i of the query rows of the keys' band
//                  windows, summed per key, added to the importance.
// The logits s' = <q * scale * log2(e), k> are formed by the same loads and
// the same FMA order in both passes, so pass 2 sees exactly pass 1's values.
// Slot j of a unit holds position j here: the host only allows the call on
// units that have been appended to and never cut.
#include "hikv_internal.cuh"

namespace hikv {
namespace {

constexpr int kBT = 64;          // query rows and keys per tile
constexpr int kBThreads = 256;   // 16 x 16 threads, 4 x 4 outputs each
constexpr int kBLd = kBT + 4;    // padded shared-memory row of a transposed tile (floats)

struct BandArgs {
    View v;
    int32_t u0;          // first unit of the layer
    int32_t li;          // the layer's index in q
    const uint8_t* q;    // [nl][B][Hq][n][d]
    int32_t n;           // tokens per unit (positions 0..n-1)
    int32_t band;        // queries per band
    float qscale;        // scale * log2(e)
    float2* stats;       // [per_layer][G][n]: (m, 1 / l) of each query row
};

// Query rows r0 .. r0 + 63 (row R = position R / G, head R % G of the
// group), scaled, transposed into Qs[c][r]; rows >= nrows are zero.
template <typename T>
__device__ void band_load_q(const BandArgs& a, int32_t ul, int32_t r0, int32_t nrows, float* Qs) {
    const int d = a.v.d, G = a.v.group;
    const int32_t b = ul / a.v.hkv, g = ul % a.v.hkv;
    const T* base = reinterpret_cast<const T*>(a.q) +
                    (((int64_t)a.li * a.v.batch + b) * a.v.hq + (int64_t)g * G) * (int64_t)a.n * d;
    for (int e = threadIdx.x; e < kBT * d; e += kBThreads) {
        const int r = e / d, c = e % d;
        const int32_t R = r0 + r;
        float x = 0.f;
        if (R < nrows) {
            const int32_t i = R / G, hh = R % G;
            x = Elem<T>::to_f(base[((int64_t)hh * a.n + i) * d + c]) * a.qscale;
        }
        Qs[c * kBLd + r] = x;
    }
}

// Keys j0 .. j0 + 63 of unit u, transposed into Ks[c][j]; keys >= n are zero.
template <typename T>
__device__ void band_load_k(const View& v, int32_t u, int32_t j0, int32_t n, float* Ks) {
    const int d = v.d;
    for (int e = threadIdx.x; e < kBT * d; e += kBThreads) {
        const int r = e / d, c = e % d;
        const int32_t j = j0 + r;
        float x = 0.f;
        if (j < n) {
            const int32_t pg = v.page_table[(int64_t)u * v.max_pages + (j >> v.page_shift)];
            if (pg >= 0 && pg < v.pool_pages) {
                const T* row = reinterpret_cast<const T*>(v.pool + (int64_t)pg * v.page_bytes +
                                                          (int64_t)(j & (v.page_tokens - 1)) * v.row_bytes);
                x = Elem<T>::to_f(row[c]);
            } else if (c == 0) {
                atomicOr(v.err, DEVERR_PAGE);
            }
        }
        Ks[c * kBLd + r] = x;
    }
}

// S[a][b] = <Qs row ty*4+a, Ks column tx*4+b>, c ascending
__device__ __forceinline__ void band_tile(const float* Qs, const float* Ks, int d, float (&S)[4][4]) {
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) S[i][j] = 0.f;
#pragma unroll 4
    for (int c = 0; c < d; ++c) {
        const float4 qa = *reinterpret_cast<const float4*>(Qs + c * kBLd + ty * 4);
        const float4 kb = *reinterpret_cast<const float4*>(Ks + c * kBLd + tx * 4);
        const float qv[4] = {qa.x, qa.y, qa.z, qa.w};
        const float kv[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) S[i][j] = fmaf(qv[i], kv[j], S[i][j]);
    }
}

template <typename T>
__global__ void __launch_bounds__(kBThreads) k_band_stats(const BandArgs a) {
    extern __shared__ float4 band_smem4[];
    const int d = a.v.d, G = a.v.group;
    float* Qs = reinterpret_cast<float*>(band_smem4);
    float* Ks = Qs + d * kBLd;
    const int32_t ul = blockIdx.y, u = a.u0 + ul;
    const int32_t n = a.n, nrows = n * G;
    const int32_t r0 = blockIdx.x * kBT;
    if (r0 >= nrows) return;
    const int32_t i_last = min(n - 1, (r0 + kBT - 1) / G);   // last query position of the tile
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    band_load_q<T>(a, ul, r0, nrows, Qs);
    float m[4], l[4];
    int32_t ipos[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int32_t R = r0 + ty * 4 + i;
        m[i] = -INFINITY;
        l[i] = 0.f;
        ipos[i] = R < nrows ? R / G : -1;   // -1: no row, every key masked
    }
    for (int32_t j0 = 0; j0 <= i_last; j0 += kBT) {
        __syncthreads();   // the previous key tile has been read
        band_load_k<T>(a.v, u, j0, n, Ks);
        __syncthreads();
        float S[4][4];
        band_tile(Qs, Ks, d, S);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float tm = -INFINITY;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (j0 + tx * 4 + j <= ipos[i]) tm = fmaxf(tm, S[i][j]);
            if (tm > -INFINITY) {
                const float nm = fmaxf(m[i], tm);
                float acc = l[i] * exp2f(m[i] - nm);   // 0 while m = -inf (l = 0)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (j0 + tx * 4 + j <= ipos[i]) acc += exp2f(S[i][j] - nm);
                m[i] = nm;
                l[i] = acc;
            }
        }
    }
    // merge the row's 16 partial states (the 16 lanes of a half warp)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float mm = m[i];
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, o));
        float ll = m[i] == -INFINITY ? 0.f : l[i] * exp2f(m[i] - mm);
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) ll += __shfl_xor_sync(0xffffffffu, ll, o);
        const int32_t R = r0 + ty * 4 + i;
        if (tx == 0 && R < nrows) {
            const int32_t pos = R / G, hh = R % G;
            a.stats[((int64_t)ul * G + hh) * n + pos] = make_float2(mm, 1.0f / ll);
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kBThreads) k_band_scores(const BandArgs a) {
    extern __shared__ float4 band_smem4[];
    const int d = a.v.d, G = a.v.group;
    float* Qs = reinterpret_cast<float*>(band_smem4);
    float* Ks = Qs + d * kBLd;
    float* Ms = Ks + d * kBLd;      // [kBT] m of the tile's rows
    float* Ls = Ms + kBT;           // [kBT] 1 / l
    float* red = Ls + kBT;          // [16][kBT] per-thread-row column sums
    const int32_t ul = blockIdx.y, u = a.u0 + ul;
    const int32_t n = a.n;
    const int32_t j0 = blockIdx.x * kBT;
    if (j0 >= n) return;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    band_load_k<T>(a.v, u, j0, n, Ks);
    // query rows whose position lies in some key's band: i in [j0, j0 + 63 + band - 1]
    const int32_t iend = (int32_t)min((int64_t)n, (int64_t)j0 + kBT - 1 + a.band);   // exclusive
    const int32_t rend = iend * G;
    float csum[4] = {0.f, 0.f, 0.f, 0.f};
    for (int32_t R0 = j0 * G; R0 < rend; R0 += kBT) {
        __syncthreads();   // the previous row tile has been read
        band_load_q<T>(a, ul, R0, rend, Qs);
        for (int r = threadIdx.x; r < kBT; r += kBThreads) {
            const int32_t R = R0 + r;
            float2 st = make_float2(0.f, 0.f);
            if (R < rend) st = a.stats[((int64_t)ul * G + R % G) * n + R / G];
            Ms[r] = st.x;
            Ls[r] = st.y;
        }
        __syncthreads();
        float S[4][4];
        band_tile(Qs, Ks, d, S);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int32_t R = R0 + ty * 4 + i;
            if (R >= rend) continue;
            const int32_t qi = R / G;
            const float mr = Ms[ty * 4 + i], li = Ls[ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int32_t kj = j0 + tx * 4 + j;
                if (kj <= qi && qi - kj < a.band) csum[j] += exp2f(S[i][j] - mr) * li;
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 4; ++j) red[ty * kBT + tx * 4 + j] = csum[j];
    __syncthreads();
    if (threadIdx.x < kBT) {
        const int32_t kj = j0 + threadIdx.x;
        if (kj < n) {
            float s = 0.f;
            for (int t = 0; t < 16; ++t) s += red[t * kBT + threadIdx.x];
            float* imp = a.v.imp + (int64_t)u * a.v.cap + kj;
            *imp = *imp + s;
        }
    }
}

size_t band_smem(int d, bool scores) {
    size_t f = 2 * (size_t)d * kBLd;
    if (scores) f += 2 * kBT + 16 * kBT;
    return f * 4;
}

template <typename T>
cudaError_t band_launch_t(const BandArgs& a, int32_t units, cudaStream_t s) {
    const size_t s1 = band_smem(a.v.d, false), s2 = band_smem(a.v.d, true);
    cudaError_t e = func_smem_optin(reinterpret_cast<const void*>(k_band_stats<T>), s1);
    if (e != cudaSuccess) return e;
    e = func_smem_optin(reinterpret_cast<const void*>(k_band_scores<T>), s2);
    if (e != cudaSuccess) return e;
    const int64_t rows = (int64_t)a.n * a.v.group;
    k_band_stats<T><<<dim3((unsigned)ceil_div((int32_t)rows, kBT), (unsigned)units), kBThreads, s1, s>>>(a);
    k_band_scores<T><<<dim3((unsigned)ceil_div(a.n, kBT), (unsigned)units), kBThreads, s2, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_band(const View& v, int32_t u0, int32_t units, int32_t li, const uint8_t* q, int32_t n,
                        int32_t band, float qscale, float2* stats, int dtype, cudaStream_t s) {
    BandArgs a{};
    a.v = v;
    a.u0 = u0;
    a.li = li;
    a.q = q;
    a.n = n;
    a.band = band;
    a.qscale = qscale;
    a.stats = stats;
    return dtype == 1 ? band_launch_t<__nv_bfloat16>(a, units, s) : band_launch_t<float>(a, units, s);
}

}  // namespace hikv
