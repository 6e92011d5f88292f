// Tile 128x256 of the GEMM ladder (one translation unit per tile).
#include "gemm_launch.cuh"
SDT_INSTANTIATE_GEMM_TILE(128, 256)
