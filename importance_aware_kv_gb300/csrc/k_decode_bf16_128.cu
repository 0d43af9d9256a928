// Decode kernel instantiations for element type __nv_bfloat16, head_dim 128.
#include "k_decode_small.cuh"
HIKV_DECODE_INSTANTIATE(__nv_bfloat16, 128, bf16_128)
