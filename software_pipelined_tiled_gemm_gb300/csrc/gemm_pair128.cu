// Kernel instance: CTA pairs computing 256 x 128 output tiles.
#include "gemm_instance.cuh"
SPGEMM_DEFINE_PAIR(128)
