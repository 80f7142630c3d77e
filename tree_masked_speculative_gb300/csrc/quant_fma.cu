// Dispatch of the quantized-KV kernels and the merge of their token-split
// partials.
//
// The merge follows the split reduction of metaltile-std
// flash_quantized_sdpa.rs: per query row M* = max_w M_w (and the sink logit),
// S* = sum_w S_w e^(M_w - M*) + e^(sink - M*), out = sum_w O_w e^(M_w - M*) / S*
// (out = O when S* = 0), written in the queries' type or f32.  M is kept in
// log2 units by the main pass, so the weights are powers of two here.
#include <type_traits>

#include "ta_internal.cuh"

namespace ta {

namespace {

constexpr float kLog2eM = 1.4426950408889634f;

template <typename T>
__device__ __forceinline__ void store_out(void *p, size_t i, float x, int out_f32) {
    if (out_f32) reinterpret_cast<float *>(p)[i] = x;
    else if constexpr (std::is_same<T, __half>::value) reinterpret_cast<__half *>(p)[i] = __float2half_rn(x);
    else reinterpret_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(x);
}

// One CTA per query row; the per-split weights are computed once into shared
// memory (128 splits at a time), then every thread sums its dimensions.
template <typename T>
__global__ void __launch_bounds__(128) quant_merge_kernel(const QuantArgs a) {
    __shared__ float s_w[128];
    __shared__ float s_red[2];
    const int q = blockIdx.x;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const float2 *ml = reinterpret_cast<const float2 *>(a.part_ml);
    const float sink = a.has_sinks ? kLog2eM * __ldg(a.sinks + (q % a.nQ)) : -INFINITY;
    if (warp == 0) {
        float m = sink;
        for (int w = lane; w < a.nwg; w += 32) m = fmaxf(m, __ldg(&ml[static_cast<size_t>(w) * a.rows + q].y));
        m = warp_max(m);
        float s = 0.0f;
        if (m != -INFINITY) {
            for (int w = lane; w < a.nwg; w += 32) {
                const float2 sm = __ldg(&ml[static_cast<size_t>(w) * a.rows + q]);
                if (sm.y != -INFINITY) s += sm.x * exp2f(sm.y - m);
            }
        }
        s = warp_sum(s);
        if (lane == 0) {
            s_red[0] = m;
            s_red[1] = (a.has_sinks && m != -INFINITY) ? s + exp2f(sink - m) : s;
        }
    }
    __syncthreads();
    const float mstar = s_red[0], sstar = s_red[1];
    const float inv = sstar > 0.0f ? 1.0f / sstar : 0.0f;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};   // dims t, t + 128, t + 256, t + 384
    for (int w0 = 0; w0 < a.nwg; w0 += 128) {
        const int n = min(128, a.nwg - w0);
        __syncthreads();
        if (t < n) {
            const float mw = __ldg(&ml[static_cast<size_t>(w0 + t) * a.rows + q].y);
            s_w[t] = (mw == -INFINITY || mstar == -INFINITY) ? 0.0f : exp2f(mw - mstar);
        }
        __syncthreads();
        for (int j = 0; j < n; ++j) {
            const float wj = s_w[j];
            const float *po = a.part_o + (static_cast<size_t>(w0 + j) * a.rows + q) * a.dim;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int d = t + 128 * k;
                if (d < a.dim) acc[k] = fmaf(__ldg(po + d), wj, acc[k]);
            }
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int d = t + 128 * k;
        if (d < a.dim) store_out<T>(a.out, static_cast<size_t>(q) * a.dim + d, acc[k] * inv, a.out_f32);
    }
}

}  // namespace

cudaError_t launch_quant_fma(const QuantArgs &a, cudaStream_t s) {
    if (a.bits == 4) return launch_quant_b4(a, s);
    if (a.bits == 8) return launch_quant_b8(a, s);
    return cudaErrorInvalidValue;
}

int quant_ctas_per_sm(int bits, int dim, int ng) {
    if (bits == 4) return quant_ctas_per_sm_b4(dim, ng);
    if (bits == 8) return quant_ctas_per_sm_b8(dim, ng);
    return 0;
}

cudaError_t launch_quant_merge(const QuantArgs &a, cudaStream_t s) {
    dim3 grid(a.rows);
    if (a.t_is_bf16) quant_merge_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(a);
    else quant_merge_kernel<__half><<<grid, 128, 0, s>>>(a);
    count_launch();
    return cudaGetLastError();
}

}  // namespace ta
