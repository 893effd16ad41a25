// The dgrad kernels whose epilogue applies GELU or SiLU backward (with or without
// the per-channel sums).
#include "dgrad_variant.cuh"

template cudaError_t cdg_dgrad_prepare_variant<2>(int, int, bool);
template cudaError_t cdg_dgrad_launch_variant<2>(const CdgParams &, int, int, bool, int, size_t, cudaStream_t);
template int cdg_dgrad_max_pairs_variant<2>(int, int, bool, size_t);
template cudaError_t cdg_dgrad_prepare_variant<3>(int, int, bool);
template cudaError_t cdg_dgrad_launch_variant<3>(const CdgParams &, int, int, bool, int, size_t, cudaStream_t);
template int cdg_dgrad_max_pairs_variant<3>(int, int, bool, size_t);
