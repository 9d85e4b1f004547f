// CUDA-core backward for dk = dv = 128 without decay: the register-tiled
// sweeps (compiled apart from the generic head-size instances).
#define LA_DK 128
#define LA_TILED128_ONLY
#include "la_simt_bwd.cuh"
