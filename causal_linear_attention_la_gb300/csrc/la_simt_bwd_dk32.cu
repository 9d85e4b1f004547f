// CUDA-core backward kernels for key head size 32.
#define LA_DK 32
#include "la_simt_bwd.cuh"
