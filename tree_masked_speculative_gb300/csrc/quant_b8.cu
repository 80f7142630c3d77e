// 8-bit instances of the quantized-KV kernel.
#include "quant_kernel.cuh"

namespace ta {
cudaError_t launch_quant_b8(const QuantArgs &a, cudaStream_t s) { return quant::launch_bits<8>(a, s); }
int quant_ctas_per_sm_b8(int dim, int ng) { return quant::occupancy_bits<8>(dim, ng); }
}  // namespace ta
