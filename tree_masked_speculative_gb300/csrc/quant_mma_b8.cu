// 8-bit instances of the warp-MMA quantized-KV kernel.
#include "quant_mma.cuh"

namespace ta {
cudaError_t launch_quant_mma_b8(const QuantArgs &a, cudaStream_t s) { return quant::mma_launch_bits<8>(a, s); }
int quant_mma_ctas_per_sm_b8(int dim, int ng) { return quant::mma_occupancy_bits<8>(dim, ng); }
}  // namespace ta
