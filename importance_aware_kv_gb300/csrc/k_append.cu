// Append (k, v) tokens to every unit of a layer range.
//
// The new token of a decode step enters the cache after the step's attention
// in HiKV's Algorithm 1; here the caller appends before hikv_decode_step so
// that the token attends to itself, as a standard decoder does.  Slots are
// the unit's next free ones (the cache stays densely packed; eviction
// compacts), pages come from the shared free stack (blog sec. 5.1: paged KV
// blocks).
#include "hikv_internal.cuh"

namespace hikv {
namespace {

// Per unit: reserve ntok slots and map the pages they need.  Writes the
// first slot to base[u - u0] (-1 when the pool ran dry, which the host's
// capacity check makes impossible).
__device__ void reserve_unit(const View& v, int32_t u, int32_t ntok, int32_t* base_out) {
    int32_t n = v.len[u];
    int32_t need = ceil_div(n + ntok, v.page_tokens);
    int32_t m = v.mapped[u];
    if (n + ntok > v.cap || need > v.max_pages) {
        atomicOr(v.err, DEVERR_STATE);
        *base_out = -1;
        return;
    }
    if (need > m) {
        int32_t cnt = need - m;
        int32_t old = atomicSub(v.free_top, cnt);
        if (old - cnt < 0) {
            atomicAdd(v.free_top, cnt);
            atomicOr(v.err, DEVERR_POOL);
            *base_out = -1;
            return;
        }
        for (int32_t i = 0; i < cnt; ++i)
            v.page_table[(int64_t)u * v.max_pages + m + i] = v.free_stack[old - cnt + i];
        v.mapped[u] = need;
    }
    *base_out = n;
    v.len[u] = n + ntok;
    v.next_pos[u] += ntok;
}

__device__ void copy_rows(const View& v, int32_t u, int32_t slot0, int32_t pos0,
                          const uint8_t* ksrc, const uint8_t* vsrc, int32_t r0, int32_t r1) {
    const int32_t vec_per_row = v.row_bytes / 16;
    const int32_t total = (r1 - r0) * vec_per_row;
    for (int32_t i = threadIdx.x; i < 2 * total; i += blockDim.x) {
        bool isv = i >= total;
        int32_t j = isv ? i - total : i;
        int32_t r = r0 + j / vec_per_row;
        int32_t c = j % vec_per_row;
        uint8_t* dst = row_ptr(v, u, slot0 + r, isv);
        if (!dst) continue;
        const uint8_t* src = (isv ? vsrc : ksrc) + (int64_t)r * v.row_bytes;
        reinterpret_cast<uint4*>(dst)[c] = __ldg(reinterpret_cast<const uint4*>(src) + c);
    }
    for (int32_t r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
        int64_t m = (int64_t)u * v.cap + slot0 + r;
        v.imp[m] = 0.0f;
        v.pos[m] = pos0 + r;
    }
}

// One CTA per unit: reserve, then copy all ntok rows (small appends).
__global__ void __launch_bounds__(256) k_append_fused(AppendArgs a) {
    __shared__ int32_t s_base, s_pos0;
    const int32_t u = a.u0 + blockIdx.x;
    if (threadIdx.x == 0) {
        int32_t b;
        reserve_unit(a.v, u, a.ntok, &b);
        s_base = b;
        s_pos0 = a.v.next_pos[u] - a.ntok;
    }
    __syncthreads();
    if (s_base < 0) return;
    const int64_t src_off = (int64_t)blockIdx.x * a.ntok * a.v.row_bytes;
    copy_rows(a.v, u, s_base, s_pos0, a.k + src_off, a.vv + src_off, 0, a.ntok);
}

// Thread per unit: reserve only (large appends).
__global__ void k_append_reserve(AppendArgs a) {
    int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= a.nunits) return;
    int32_t b;
    reserve_unit(a.v, a.u0 + i, a.ntok, &b);
    a.base[i] = b;
}

constexpr int kRowsPerCta = 64;

// grid (row blocks, units): copy a block of rows after k_append_reserve.
__global__ void __launch_bounds__(256) k_append_copy(AppendArgs a) {
    const int32_t i = blockIdx.y;
    const int32_t u = a.u0 + i;
    const int32_t base = a.base[i];
    if (base < 0) return;
    const int32_t pos0 = a.v.next_pos[u] - a.ntok;
    const int32_t r0 = blockIdx.x * kRowsPerCta;
    const int32_t r1 = min(a.ntok, r0 + kRowsPerCta);
    const int64_t src_off = (int64_t)i * a.ntok * a.v.row_bytes;
    copy_rows(a.v, u, base, pos0, a.k + src_off, a.vv + src_off, r0, r1);
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s) {
    if (a.nunits <= 0 || a.ntok <= 0) return cudaSuccess;
    if (a.ntok <= kRowsPerCta) {
        k_append_fused<<<a.nunits, 256, 0, s>>>(a);
        return cudaGetLastError();
    }
    k_append_reserve<<<ceil_div(a.nunits, 128), 128, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 grid(ceil_div(a.ntok, kRowsPerCta), a.nunits);
    k_append_copy<<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace hikv
