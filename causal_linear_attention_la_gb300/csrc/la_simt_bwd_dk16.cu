// CUDA-core backward kernels for key head size 16.
#define LA_DK 16
#include "la_simt_bwd.cuh"
