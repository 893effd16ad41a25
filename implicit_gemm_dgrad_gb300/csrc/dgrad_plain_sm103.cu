// The dgrad kernels with the plain epilogue (the ReLU gate or none): what every
// default plan launches.
#include "dgrad_variant.cuh"

template cudaError_t cdg_dgrad_prepare_variant<0>(int, int, bool);
template cudaError_t cdg_dgrad_launch_variant<0>(const CdgParams &, int, int, bool, int, size_t, cudaStream_t);
template int cdg_dgrad_max_pairs_variant<0>(int, int, bool, size_t);
