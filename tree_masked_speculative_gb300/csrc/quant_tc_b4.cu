// 4-bit instances of the tensor-core quantized-KV kernel (quant_tc.cuh).
#include "quant_tc.cuh"

namespace ta {

cudaError_t launch_quant_tc_b4(const QuantArgs &a, size_t smem, cudaStream_t s) {
    return qtc::launch_bits<4>(a, smem, s);
}

int quant_tc_ctas_per_sm_b4(int rp, size_t smem) { return qtc::occupancy_bits<4>(rp, smem); }

}  // namespace ta
