// CUDA-core forward kernels for key head size 128.
#define LA_DK 128
#include "la_simt_fwd.cuh"
