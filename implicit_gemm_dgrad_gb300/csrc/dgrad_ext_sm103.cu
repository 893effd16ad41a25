// The dgrad kernels with the extended epilogue (per-channel sums, activation
// backward other than ReLU), instantiated for plans that ask for it.
#include "dgrad_variant.cuh"

template cudaError_t cdg_dgrad_prepare_variant<true>(int, int, bool);
template cudaError_t cdg_dgrad_launch_variant<true>(const CdgParams &, int, int, bool, int, size_t, cudaStream_t);
template int cdg_dgrad_max_pairs_variant<true>(int, int, bool, size_t);
