// Placeholder until the tcgen05 kernels land: every case runs the fp32 kernels.
#include "internal.h"

namespace flashbob {
bool tc_supported(const BobArgs&) { return false; }
cudaError_t tc_bob(const BobArgs&) { return cudaErrorNotSupported; }
size_t tc_pass1_smem() { return 0; }
size_t tc_pass2_smem() { return 0; }
}  // namespace flashbob
