// Dispatch of the fused decode kernel over (dtype, head_dim).
#include "hikv_internal.cuh"

namespace hikv {

#define HIKV_DECL(NAME)                                                                            \
    cudaError_t decode_launch_##NAME(const DecodeArgs&, const CUtensorMap&, int, bool, size_t, cudaStream_t); \
    size_t decode_smem_##NAME(int, bool, int);                                                     \
    int decode_active_##NAME(int, bool, int, size_t);                                               \
    cudaError_t decode_small_launch_##NAME(const SmallArgs&, const CUtensorMap&, int, int, cudaStream_t);
HIKV_DECL(f32_64)
HIKV_DECL(f32_128)
HIKV_DECL(bf16_64)
HIKV_DECL(bf16_128)
#undef HIKV_DECL

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& tmap, int dtype, int d, int group,
                          bool smem_path, size_t smem_bytes, cudaStream_t s) {
    if (dtype == 0 && d == 64) return decode_launch_f32_64(a, tmap, group, smem_path, smem_bytes, s);
    if (dtype == 0 && d == 128) return decode_launch_f32_128(a, tmap, group, smem_path, smem_bytes, s);
    if (dtype == 1 && d == 64) return decode_launch_bf16_64(a, tmap, group, smem_path, smem_bytes, s);
    if (dtype == 1 && d == 128) return decode_launch_bf16_128(a, tmap, group, smem_path, smem_bytes, s);
    return cudaErrorInvalidValue;
}

size_t decode_smem_bytes(int dtype, int d, int group, bool smem_path, int chunk_cap) {
    if (dtype == 0 && d == 64) return decode_smem_f32_64(group, smem_path, chunk_cap);
    if (dtype == 0 && d == 128) return decode_smem_f32_128(group, smem_path, chunk_cap);
    if (dtype == 1 && d == 64) return decode_smem_bf16_64(group, smem_path, chunk_cap);
    if (dtype == 1 && d == 128) return decode_smem_bf16_128(group, smem_path, chunk_cap);
    return 0;
}

int decode_active_clusters(int dtype, int d, int group, bool smem_path, int cs, size_t smem_bytes) {
    if (dtype == 0 && d == 64) return decode_active_f32_64(group, smem_path, cs, smem_bytes);
    if (dtype == 0 && d == 128) return decode_active_f32_128(group, smem_path, cs, smem_bytes);
    if (dtype == 1 && d == 64) return decode_active_bf16_64(group, smem_path, cs, smem_bytes);
    if (dtype == 1 && d == 128) return decode_active_bf16_128(group, smem_path, cs, smem_bytes);
    return 0;
}

cudaError_t launch_decode_small(const SmallArgs& a, const CUtensorMap& tmap, int dtype, int d, int group,
                                int n_ctas, cudaStream_t s) {
    if (dtype == 0 && d == 64) return decode_small_launch_f32_64(a, tmap, group, n_ctas, s);
    if (dtype == 0 && d == 128) return decode_small_launch_f32_128(a, tmap, group, n_ctas, s);
    if (dtype == 1 && d == 64) return decode_small_launch_bf16_64(a, tmap, group, n_ctas, s);
    if (dtype == 1 && d == 128) return decode_small_launch_bf16_128(a, tmap, group, n_ctas, s);
    return cudaErrorInvalidValue;
}

// Largest chunk (tokens per CTA) whose logits fit the shared-memory path.
int decode_max_smem_chunk(int dtype, int d, int group, size_t smem_limit) {
    int lo = 0, hi = 1 << 16;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (decode_smem_bytes(dtype, d, group, true, mid) <= smem_limit) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

}  // namespace hikv
