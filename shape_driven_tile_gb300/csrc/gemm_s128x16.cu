// Skinny tile 128x16 (operands swapped; gemm_ex forms only), one translation unit.
#include "gemm_launch.cuh"
SDT_INSTANTIATE_GEMM_TILE(128, 16)
