// 8-bit instances of the wide (16 query rows per warp) warp-MMA quantized-KV kernel.
#include "quant_mma16.cuh"

namespace ta {
cudaError_t launch_quant_mma16_b8(const QuantArgs &a, cudaStream_t s) { return quant::mma16_launch_bits<8>(a, s); }
int quant_mma16_ctas_per_sm_b8(int dim, int ng) { return quant::mma16_occupancy_bits<8>(dim, ng); }
}  // namespace ta
