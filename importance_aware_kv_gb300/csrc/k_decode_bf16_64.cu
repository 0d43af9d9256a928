// Decode kernel instantiations for element type __nv_bfloat16, head_dim 64.
#include "k_decode_small.cuh"
HIKV_DECODE_INSTANTIATE(__nv_bfloat16, 64, bf16_64)
