// Decode kernel instantiations for element type float, head_dim 128.
#include "k_decode_small.cuh"
HIKV_DECODE_INSTANTIATE(float, 128, f32_128)
