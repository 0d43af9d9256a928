// SnapKV pooling of the prompt scores (setup step).
//
// SnapKV keeps prefix tokens by their observation-window score max-pooled
// along the sequence, S_pooled[i] = max_{0<=m<k} A_obs[i+m], so that a whole
// phrase around a salient token survives (KV cache compression blog, sec. 3
// "SnapKV").  Applied to the window scores left by hikv_score_window while a
// unit still holds its whole prompt in position order (slot s = position s);
// positions past the unit's end contribute nothing.
//
// One CTA per unit walks its slots in chunks of kPoolChunk, in increasing
// order: a chunk reads its k - 1 halo slots from the next chunk before that
// chunk is rewritten, so the pooling runs in place.
#include "hikv_internal.cuh"

namespace hikv {
namespace {

constexpr int kPoolThreads = 256;
constexpr int kPoolChunk = 2048;

__global__ void __launch_bounds__(kPoolThreads) k_pool_importance(View v, int32_t u0, int32_t k) {
    __shared__ float buf[kPoolChunk + kMaxPoolKernel];
    const int32_t u = u0 + blockIdx.x;
    const int32_t n = v.len[u];
    float* imp = v.imp + (int64_t)u * v.cap;
    const int32_t* pos = v.pos + (int64_t)u * v.cap;
    for (int32_t c0 = 0; c0 < n; c0 += kPoolChunk) {
        const int32_t c1 = min(n, c0 + kPoolChunk);
        const int32_t h1 = min(n, c1 + k - 1);   // halo end
        for (int32_t s = c0 + threadIdx.x; s < h1; s += kPoolThreads) {
            buf[s - c0] = imp[s];
            if (pos[s] != s) atomicOr(v.err, DEVERR_STATE);   // not the uncut prompt
        }
        __syncthreads();
        for (int32_t s = c0 + threadIdx.x; s < c1; s += kPoolThreads) {
            const int32_t e = min(h1, s + k);
            float m = buf[s - c0];
            for (int32_t j = s + 1; j < e; ++j) m = fmaxf(m, buf[j - c0]);
            imp[s] = m;
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_pool_importance(const View& v, int32_t u0, int32_t nu, int k, cudaStream_t s) {
    if (nu <= 0 || k <= 1) return cudaSuccess;
    k_pool_importance<<<nu, kPoolThreads, 0, s>>>(v, u0, k);
    return cudaGetLastError();
}

}  // namespace hikv
