// Decode kernel instantiations for element type float, head_dim 64.
#include "k_decode_small.cuh"
HIKV_DECODE_INSTANTIATE(float, 64, f32_64)
