// Kernel instance: 128 x 128 output tiles.
#include "gemm_instance.cuh"
SPGEMM_DEFINE_BN(128)
