// hca_tc.cu -- tensor-core (tcgen05) HCA kernels (placeholder: not yet built).
#include "hca_common.cuh"
#include "hca_internal.h"

namespace hca {
bool tc_fwd_supported(int, int, int) { return false; }
int tc_query_tile_positions(int) { return 1; }
cudaError_t tc_fwd(const FwdArgs &, cudaStream_t) { return cudaErrorNotSupported; }
bool tc_bwd_supported(int, int, int) { return false; }
size_t tc_bwd_scratch_bytes(int, int, int, int, int, int, int) { return 0; }
cudaError_t tc_bwd(const BwdArgs &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace hca
