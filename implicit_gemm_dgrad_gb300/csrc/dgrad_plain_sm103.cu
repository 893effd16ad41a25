// The dgrad kernels without the extended epilogue (per-channel sums, activation
// backward other than ReLU): the plain kernels every default plan launches.
#include "dgrad_variant.cuh"

template cudaError_t cdg_dgrad_prepare_variant<false>(int, int, bool);
template cudaError_t cdg_dgrad_launch_variant<false>(const CdgParams &, int, int, bool, int, size_t, cudaStream_t);
template int cdg_dgrad_max_pairs_variant<false>(int, int, bool, size_t);
