// correlate_bank_tc.cu -- template-bank correlation on the tensor cores
// (placeholder until the tcgen05 kernel lands: banks run template by
// template on the dp4a kernel).
#include "ncc_common.cuh"

namespace ncc {

bool bank_tc_supported(int, int, int, int, int) { return false; }

cudaError_t bank_tc_launch(const BankArgs &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace ncc
