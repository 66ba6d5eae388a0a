// Kernel instance: 128 x 64 output tiles.
#include "gemm_instance.cuh"
SPGEMM_DEFINE_BN(64)
