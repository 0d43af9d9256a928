// Prefill window scoring for callers that cannot allocate device memory.
//
// hikv_score_window computes prompt importance inside a cache, whose work
// buffers come from cudaMalloc at hikv_create_cache.  Some callers cannot
// call cudaMalloc at all: plugins running inside an inference engine that owns
// every device allocation and forbids allocating while it executes, or code
// on a real-time path where an allocation (and the device synchronisation it
// may imply) is not allowed.  For them this file offers the same computation
// as a stateless call on buffers the caller already owns: keys of the prompt
// in, importance out.  Its only scratch -- the per-chunk partial (max, sum) of
// every query vector -- lives in a file-scope static __device__ array, which
// the CUDA runtime creates when the module loads and keeps until the process
// exits, on every device that loads this library.
//
// The arithmetic is the two-pass scheme of the cache's window scoring: pass 1
// reduces each 1024-token chunk to a partial (max, sum of 2^(s' - max)) per
// query vector; pass 2 merges the partials and adds, query by query in
// position order, sum_h 2^(s' - m) / l to every token the query may see
// (causal: token position <= query position).  Token j of a unit has
// position j; the queries are those of the last nq positions.
#include <cmath>
#include <cstdio>
#include <mutex>

#include "../../include/hikv.h"
#include "hikv_internal.cuh"

namespace hikv {
namespace {

constexpr int kNaThreads = 256;
constexpr int kNaTT = 32;     // tokens per sub-tile
constexpr int kNaQB = 64;     // query vectors per block
constexpr int kNaChunk = 1024;
constexpr int64_t kNaScratchFloats = 1 << 20;   // 4 MiB of partial (max, sum) pairs
constexpr int kNaMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_part[kNaScratchFloats];

struct NaArgs {
    const uint8_t* k;     // [units][ntok][d]
    const uint8_t* q;     // [nl][B][Hq][nq][d]
    float* imp;           // [units][ntok]
    float* part;          // [units][nch][nqv][2] inside g_noalloc_part
    int32_t units, batch, hq, hkv, group, d, ntok, nq, nch;
    float qscale;
};

template <typename T>
__device__ void na_load_k(const NaArgs& a, int32_t u, int32_t s0, int32_t s1, float* Ks) {
    const int d = a.d;
    const T* base = reinterpret_cast<const T*>(a.k) + (int64_t)u * a.ntok * d;
    for (int i = threadIdx.x; i < kNaTT * d; i += kNaThreads) {
        const int r = i / d, c = i % d;
        const int32_t s = s0 + r;
        Ks[r * (d + 1) + c] = (s < s1) ? Elem<T>::to_f(base[(int64_t)s * d + c]) : 0.f;
    }
}

__device__ void na_tile_logits(const float* Ks, const float* Qs, int d, int qb, int nqv, float* St) {
    const int tq = threadIdx.x % 16, tt = threadIdx.x / 16;
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
        for (int j = 0; j < 4; ++j) St[(tt * 2 + r) * kNaQB + tq * 4 + j] = acc[r][j];
}

template <typename T>
__device__ void na_load_q(const NaArgs& a, int32_t u, float* Qs) {
    const int d = a.d, G = a.group, nq = a.nq;
    const int32_t per_layer = a.batch * a.hkv;
    const int32_t li = u / per_layer, b = (u / a.hkv) % a.batch, g = u % a.hkv;
    const T* base = reinterpret_cast<const T*>(a.q) + (((int64_t)li * a.batch + b) * a.hq + (int64_t)g * G) * nq * d;
    for (int i = threadIdx.x; i < G * nq * d; i += kNaThreads) {
        const int qv = i / d, c = i % d;
        Qs[qv * (d + 1) + c] = Elem<T>::to_f(base[(int64_t)qv * d + c]) * a.qscale;
    }
}

template <typename T>
__global__ void __launch_bounds__(kNaThreads) k_na_p1(NaArgs a) {
    extern __shared__ float wsm[];
    const int d = a.d, nqv = a.group * a.nq;
    const int32_t u = blockIdx.y;
    const int32_t c0 = blockIdx.x * kNaChunk, c1 = min(a.ntok, c0 + kNaChunk);
    const int32_t tnew = a.ntok - 1;
    float* part = a.part + (((int64_t)u * a.nch + blockIdx.x) * nqv) * 2;
    float* Qs = wsm;
    float* Ks = Qs + nqv * (d + 1);
    float* St = Ks + kNaTT * (d + 1);
    float* ML = St + kNaTT * kNaQB;   // [nqv][2]
    na_load_q<T>(a, u, Qs);
    for (int q = threadIdx.x; q < nqv; q += kNaThreads) {
        ML[2 * q] = -INFINITY;
        ML[2 * q + 1] = 0.f;
    }
    for (int32_t s0 = c0; s0 < c1; s0 += kNaTT) {
        __syncthreads();
        na_load_k<T>(a, u, s0, c1, Ks);
        __syncthreads();
        for (int qb = 0; qb < nqv; qb += kNaQB) {
            na_tile_logits(Ks, Qs, d, qb, nqv, St);
            __syncthreads();
            const int q = qb + threadIdx.x;
            if (threadIdx.x < kNaQB && q < nqv) {
                const int32_t qpos = tnew - a.nq + 1 + q % a.nq;
                float m = ML[2 * q], l = ML[2 * q + 1];
                float tm = -INFINITY;
                for (int r = 0; r < kNaTT; ++r)
                    if (s0 + r < c1 && s0 + r <= qpos) tm = fmaxf(tm, St[r * kNaQB + threadIdx.x]);
                if (tm > -INFINITY) {
                    const float nm = fmaxf(m, tm);
                    float acc = (l > 0.f) ? l * exp2f(m - nm) : 0.f;
                    for (int r = 0; r < kNaTT; ++r)
                        if (s0 + r < c1 && s0 + r <= qpos) acc += exp2f(St[r * kNaQB + threadIdx.x] - nm);
                    ML[2 * q] = nm;
                    ML[2 * q + 1] = acc;
                }
            }
            __syncthreads();
        }
    }
    __syncthreads();
    for (int q = threadIdx.x; q < nqv; q += kNaThreads) {
        part[2 * q] = ML[2 * q];
        part[2 * q + 1] = ML[2 * q + 1];
    }
}

template <typename T>
__global__ void __launch_bounds__(kNaThreads) k_na_p2(NaArgs a) {
    extern __shared__ float wsm[];
    const int d = a.d, G = a.group, nq = a.nq, nqv = G * nq;
    const int32_t u = blockIdx.y;
    const int32_t c0 = blockIdx.x * kNaChunk, c1 = min(a.ntok, c0 + kNaChunk);
    const int32_t tnew = a.ntok - 1;
    float* Qs = wsm;
    float* Ks = Qs + nqv * (d + 1);
    float* St = Ks + kNaTT * (d + 1);
    float* MF = St + kNaTT * kNaQB;   // [nqv]
    float* LI = MF + nqv;             // [nqv]
    float* Pt = LI + nqv;             // [TT][nqv]
    na_load_q<T>(a, u, Qs);
    const float* part = a.part + ((int64_t)u * a.nch) * nqv * 2;
    for (int q = threadIdx.x; q < nqv; q += kNaThreads) {
        float m = -INFINITY;
        for (int cc = 0; cc < a.nch; ++cc) m = fmaxf(m, part[((int64_t)cc * nqv + q) * 2]);
        float l = 0.f;
        for (int cc = 0; cc < a.nch; ++cc) {
            const float lc = part[((int64_t)cc * nqv + q) * 2 + 1];
            if (lc > 0.f) l += lc * exp2f(part[((int64_t)cc * nqv + q) * 2] - m);
        }
        MF[q] = m;
        LI[q] = 1.0f / l;
    }
    for (int32_t s0 = c0; s0 < c1; s0 += kNaTT) {
        __syncthreads();
        na_load_k<T>(a, u, s0, c1, Ks);
        __syncthreads();
        for (int qb = 0; qb < nqv; qb += kNaQB) {
            na_tile_logits(Ks, Qs, d, qb, nqv, St);
            __syncthreads();
            for (int i = threadIdx.x; i < kNaTT * kNaQB; i += kNaThreads) {
                const int r = i / kNaQB, qq = i % kNaQB, q = qb + qq;
                if (q >= nqv) continue;
                const int32_t qpos = tnew - nq + 1 + q % nq;
                Pt[r * nqv + q] = (s0 + r <= qpos) ? exp2f(St[r * kNaQB + qq] - MF[q]) * LI[q] : 0.f;
            }
            __syncthreads();
        }
        for (int r = threadIdx.x; r < kNaTT; r += kNaThreads) {
            const int32_t s = s0 + r;
            if (s >= c1) continue;
            float imp = 0.f;   // a fresh prompt token starts at importance 0
            for (int i = 0; i < nq; ++i) {
                float inc = 0.f;
                for (int hh = 0; hh < G; ++hh) inc += Pt[r * nqv + hh * nq + i];
                imp = imp + inc;
            }
            a.imp[(int64_t)u * a.ntok + s] = imp;
        }
    }
}

size_t na_smem(int d, int nqv) {
    size_t f = (size_t)nqv * (d + 1) + (size_t)kNaTT * (d + 1) + (size_t)kNaTT * kNaQB;
    f += 2 * (size_t)nqv + (size_t)kNaTT * nqv;
    return f * 4;
}

// device address of the static scratch, looked up once per device
float* g_part_ptr[kNaMaxDevices] = {};
std::mutex g_part_mu;

}  // namespace

void set_last_error(const char* msg);   // hikv_last_error() reports it

namespace {
hikv_status na_fail(hikv_status s, const char* msg) {
    set_last_error(msg);
    return s;
}
}  // namespace
}  // namespace hikv

using namespace hikv;

extern "C" hikv_status hikv_score_window_noalloc(int32_t nlayers, int32_t batch, int32_t num_q_heads,
                                                 int32_t num_kv_heads, int32_t head_dim, int32_t dtype,
                                                 int32_t ntok, int32_t nq, float scale, const void* k,
                                                 const void* q, float* importance, hikv_stream_t stream) {
    set_last_error("");
    if (nlayers <= 0 || batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || ntok <= 0 || nq <= 0)
        return na_fail(HIKV_ERR_INVALID_ARG, "score_window_noalloc: sizes must be positive");
    if (num_q_heads % num_kv_heads)
        return na_fail(HIKV_ERR_INVALID_ARG, "score_window_noalloc: num_q_heads must be a multiple of num_kv_heads");
    const int G = num_q_heads / num_kv_heads;
    if ((head_dim != 64 && head_dim != 128) || (dtype != HIKV_F32 && dtype != HIKV_BF16))
        return na_fail(HIKV_ERR_UNSUPPORTED, "score_window_noalloc: head_dim must be 64/128, dtype f32/bf16");
    if (nq > ntok) return na_fail(HIKV_ERR_INVALID_ARG, "score_window_noalloc: nq exceeds ntok");
    if (!k || !q || !importance) return na_fail(HIKV_ERR_INVALID_ARG, "score_window_noalloc: null pointer");
    if (!(scale >= 0.f)) return na_fail(HIKV_ERR_INVALID_ARG, "score_window_noalloc: bad scale");
    const int64_t units = (int64_t)nlayers * batch * num_kv_heads;
    const int nch = (ntok + kNaChunk - 1) / kNaChunk;
    const int nqv = G * nq;
    if (units > 65535)
        return na_fail(HIKV_ERR_INVALID_ARG, "score_window_noalloc: more than 65535 units");
    if (units * nch * nqv * 2 > kNaScratchFloats) {
        char buf[200];
        snprintf(buf, sizeof buf,
                 "score_window_noalloc: needs %lld scratch floats (units x ceil(ntok/1024) x G*nq x 2), "
                 "the static scratch holds %lld",
                 (long long)(units * nch * nqv * 2), (long long)kNaScratchFloats);
        return na_fail(HIKV_ERR_INVALID_ARG, buf);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kNaMaxDevices)
        return na_fail(HIKV_ERR_CUDA, "score_window_noalloc: no usable current device");
    float* part = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_part_mu);
        if (!g_part_ptr[dev]) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_part);
            if (e != cudaSuccess) return na_fail(HIKV_ERR_CUDA, "score_window_noalloc: cudaGetSymbolAddress failed");
            g_part_ptr[dev] = static_cast<float*>(p);
        }
        part = g_part_ptr[dev];
    }
    const size_t smem = na_smem(head_dim, nqv);
    int optin = 0;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (smem > (size_t)optin)
        return na_fail(HIKV_ERR_UNSUPPORTED, "score_window_noalloc: G*nq query vectors exceed shared memory");
    NaArgs a{};
    a.k = (const uint8_t*)k;
    a.q = (const uint8_t*)q;
    a.imp = importance;
    a.part = part;
    a.units = (int32_t)units;
    a.batch = batch;
    a.hq = num_q_heads;
    a.hkv = num_kv_heads;
    a.group = G;
    a.d = head_dim;
    a.ntok = ntok;
    a.nq = nq;
    a.nch = nch;
    const float sc = scale > 0.f ? scale : 1.0f / sqrtf((float)head_dim);
    a.qscale = sc * 1.4426950408889634f;
    dim3 grid(nch, (unsigned)units);
    cudaStream_t s = (cudaStream_t)stream;
    if (dtype == HIKV_F32) {
        if ((e = func_smem_optin(reinterpret_cast<const void*>(k_na_p1<float>), smem)) ||
            (e = func_smem_optin(reinterpret_cast<const void*>(k_na_p2<float>), smem)))
            return na_fail(HIKV_ERR_CUDA, "score_window_noalloc: cudaFuncSetAttribute failed");
        k_na_p1<float><<<grid, kNaThreads, smem, s>>>(a);
        k_na_p2<float><<<grid, kNaThreads, smem, s>>>(a);
    } else {
        if ((e = func_smem_optin(reinterpret_cast<const void*>(k_na_p1<__nv_bfloat16>), smem)) ||
            (e = func_smem_optin(reinterpret_cast<const void*>(k_na_p2<__nv_bfloat16>), smem)))
            return na_fail(HIKV_ERR_CUDA, "score_window_noalloc: cudaFuncSetAttribute failed");
        k_na_p1<__nv_bfloat16><<<grid, kNaThreads, smem, s>>>(a);
        k_na_p2<__nv_bfloat16><<<grid, kNaThreads, smem, s>>>(a);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return na_fail(HIKV_ERR_CUDA, "score_window_noalloc: launch failed");
    return HIKV_OK;
}
