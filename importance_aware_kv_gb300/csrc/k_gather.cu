// Export of the retained state, per unit, in ascending original position.
//
// Slots are unordered (eviction moves tokens into freed slots; attention does
// not care, Kelle summary sec. 2.2), so the export ranks each slot by its
// position: positions are unique in [0, next_pos), so a bitmap of present
// positions and a prefix count over its words give every slot its rank
// directly.  The bitmap covers 2^16 positions at a time.
#include <algorithm>

#include "hikv_internal.cuh"

namespace hikv {
namespace {

constexpr int kGaThreads = 256;
constexpr int kGaWin = 1 << 16;           // positions per window
constexpr int kGaWords = kGaWin / 32;     // 2048
constexpr int kGaPer = kGaWords / kGaThreads;

__global__ void __launch_bounds__(kGaThreads) k_gather(GatherArgs a) {
    __shared__ uint32_t bm[kGaWords];
    __shared__ int32_t pre[kGaWords];
    __shared__ int32_t tsum[kGaThreads];
    const View& v = a.v;
    const int32_t i = blockIdx.x;
    const int32_t u = a.u0 + i;
    const int32_t n = v.len[u];
    const int32_t np = v.next_pos[u];
    const int64_t ob = (int64_t)i * a.cap;
    const int32_t* pos = v.pos + (int64_t)u * v.cap;
    const float* imp = v.imp + (int64_t)u * v.cap;
    const int32_t vec = v.row_bytes / 16;
    if (threadIdx.x == 0) a.lengths[i] = n;
    int32_t base = 0;
    for (int32_t w0 = 0; w0 < np; w0 += kGaWin) {
        for (int k = threadIdx.x; k < kGaWords; k += kGaThreads) bm[k] = 0;
        __syncthreads();
        for (int32_t s = threadIdx.x; s < n; s += kGaThreads) {
            const int32_t p = pos[s] - w0;
            if (p >= 0 && p < kGaWin) atomicOr(&bm[p >> 5], 1u << (p & 31));
        }
        __syncthreads();
        int32_t loc = 0;
        for (int k = 0; k < kGaPer; ++k) loc += __popc(bm[threadIdx.x * kGaPer + k]);
        tsum[threadIdx.x] = loc;
        __syncthreads();
        if (threadIdx.x == 0) {
            int32_t acc = 0;
            for (int t = 0; t < kGaThreads; ++t) {
                const int32_t x = tsum[t];
                tsum[t] = acc;
                acc += x;
            }
        }
        __syncthreads();
        {
            int32_t acc = tsum[threadIdx.x];
            for (int k = 0; k < kGaPer; ++k) {
                const int w = threadIdx.x * kGaPer + k;
                pre[w] = acc;
                acc += __popc(bm[w]);
            }
        }
        __syncthreads();
        for (int32_t s = threadIdx.x; s < n; s += kGaThreads) {
            const int32_t p = pos[s] - w0;
            if (p < 0 || p >= kGaWin) continue;
            const int32_t r = base + pre[p >> 5] + __popc(bm[p >> 5] & ((1u << (p & 31)) - 1u));
            if (r >= a.cap) continue;
            a.positions[ob + r] = pos[s];
            a.importance[ob + r] = imp[s];
            for (int isv = 0; isv < 2; ++isv) {
                uint8_t* dst = isv ? a.v_out : a.k_out;
                if (!dst) continue;
                const uint8_t* src = row_ptr(v, u, s, isv != 0);
                uint4* d4 = reinterpret_cast<uint4*>(dst + (ob + r) * v.row_bytes);
                for (int32_t c = 0; c < vec; ++c) d4[c] = src ? reinterpret_cast<const uint4*>(src)[c] : make_uint4(0, 0, 0, 0);
            }
        }
        // total present in this window
        __syncthreads();
        if (threadIdx.x == 0) tsum[0] = pre[kGaWords - 1] + __popc(bm[kGaWords - 1]);
        __syncthreads();
        base += tsum[0];
        __syncthreads();
    }
    for (int32_t r = n + threadIdx.x; r < a.cap; r += kGaThreads) {
        a.positions[ob + r] = -1;
        a.importance[ob + r] = 0.f;
        for (int isv = 0; isv < 2; ++isv) {
            uint8_t* dst = isv ? a.v_out : a.k_out;
            if (!dst) continue;
            uint4* d4 = reinterpret_cast<uint4*>(dst + (ob + r) * v.row_bytes);
            for (int32_t c = 0; c < vec; ++c) d4[c] = make_uint4(0, 0, 0, 0);
        }
    }
}

}  // namespace

cudaError_t launch_gather(const GatherArgs& a, cudaStream_t s) {
    if (a.nunits <= 0) return cudaSuccess;
    k_gather<<<a.nunits, kGaThreads, 0, s>>>(a);
    return cudaGetLastError();
}

// Failure-detection self-test: one CTA waits, bounded by limit_ns, on an
// mbarrier that nothing arrives on; the wait gives up, records the timeout
// (site kWaitSelftest) in the device error word and the kernel returns, so
// the context stays usable.  No trap, no unbounded spin.
__global__ void k_selftest_timeout(View v, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        mbar_wait_bounded(&bar, 0u, v.err, kWaitSelftest, 0u, limit_ns);   // phase 0 never completes
    }
}

cudaError_t launch_selftest_timeout(const View& v, uint64_t limit_ns, cudaStream_t s) {
    k_selftest_timeout<<<1, 32, 0, s>>>(v, limit_ns);
    return cudaGetLastError();
}

namespace {
__global__ void k_fill_u32(uint32_t* p, size_t n, uint32_t word) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        p[i] = word;
}
}  // namespace

cudaError_t launch_fill_u32(uint32_t* p, size_t n, uint32_t word, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const size_t blocks = std::min<size_t>((n + 255) / 256, 65536);
    k_fill_u32<<<(unsigned)blocks, 256, 0, s>>>(p, n, word);
    return cudaGetLastError();
}

}  // namespace hikv
