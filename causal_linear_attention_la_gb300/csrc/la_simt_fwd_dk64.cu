// CUDA-core forward kernels for key head size 64.
#define LA_DK 64
#include "la_simt_fwd.cuh"
