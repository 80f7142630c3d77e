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

// One CTA per query row.  Thread t takes float4 column (t % D4) of the splits
// w = t / D4 (mod groups): its (S, M) and O loads are issued together and
// merged against the thread's own running max (log2 units); the groups, and
// the sink, are combined in shared memory.  Launched as a programmatic
// dependent of the main pass.
constexpr int kMergeThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kMergeThreads) quant_merge_kernel(const QuantArgs a) {
    pdl_wait();
    __shared__ float4 s_acc[kMergeThreads];
    __shared__ float2 s_ms[kMergeThreads];
    const int q = blockIdx.x;
    const int t = threadIdx.x;
    const int D4 = a.dim / 4;
    const int groups = kMergeThreads / D4;
    const int g = t / D4, i = t % D4;
    const float2 *ml = reinterpret_cast<const float2 *>(a.part_ml) + q;   // (S, M), stride rows
    float m = -INFINITY, ssum = 0.0f;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (g < groups) {
        const size_t stride = static_cast<size_t>(a.rows) * a.dim;
        const float *po = a.part_o + static_cast<size_t>(q) * a.dim + 4 * i;
        auto merge = [&](float2 sm, float4 o) {
            if (sm.y == -INFINITY) return;   // a split that saw no token
            const float mn = fmaxf(m, sm.y);
            const float c = exp2f(m - mn), e = exp2f(sm.y - mn);   // c = 0 while m = -inf
            m = mn;
            ssum = ssum * c + sm.x * e;
            acc.x = acc.x * c + o.x * e; acc.y = acc.y * c + o.y * e;
            acc.z = acc.z * c + o.z * e; acc.w = acc.w * c + o.w * e;
        };
        // the thread's first kPre slots are all loaded before any is merged (one round
        // trip for up to kPre * groups splits), the rest four at a time
        constexpr int kPre = 8;
        float2 sm_pre[kPre];
        float4 o_pre[kPre];
#pragma unroll
        for (int k = 0; k < kPre; ++k) {
            const int w = g + k * groups;
            if (w < a.nwg) {
                sm_pre[k] = __ldg(ml + static_cast<size_t>(w) * a.rows);
                o_pre[k] = __ldg(reinterpret_cast<const float4 *>(po + w * stride));
            }
        }
#pragma unroll
        for (int k = 0; k < kPre; ++k)
            if (g + k * groups < a.nwg) merge(sm_pre[k], o_pre[k]);
#pragma unroll 4
        for (int w = g + kPre * groups; w < a.nwg; w += groups)
            merge(__ldg(ml + static_cast<size_t>(w) * a.rows), __ldg(reinterpret_cast<const float4 *>(po + w * stride)));
    }
    s_acc[t] = acc;
    s_ms[t] = make_float2(m, ssum);
    __syncthreads();
    if (t < D4) {
        const float sink = a.has_sinks ? kLog2eM * __ldg(a.sinks + (q % a.nQ)) : -INFINITY;
        float mstar = sink;
        for (int k = 0; k < groups; ++k) mstar = fmaxf(mstar, s_ms[k * D4 + t].x);
        float sstar = 0.0f;
        float4 r = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (mstar != -INFINITY) {
            if (a.has_sinks) sstar = exp2f(sink - mstar);
            for (int k = 0; k < groups; ++k) {
                const float2 ms = s_ms[k * D4 + t];
                if (ms.x == -INFINITY) continue;
                const float w = exp2f(ms.x - mstar);
                const float4 x = s_acc[k * D4 + t];
                sstar += ms.y * w;
                r.x += x.x * w; r.y += x.y * w; r.z += x.z * w; r.w += x.w * w;
            }
        }
        const float inv = sstar > 0.0f ? 1.0f / sstar : 0.0f;
        const size_t o = static_cast<size_t>(q) * a.dim + 4 * t;
        store_out<T>(a.out, o + 0, r.x * inv, a.out_f32);
        store_out<T>(a.out, o + 1, r.y * inv, a.out_f32);
        store_out<T>(a.out, o + 2, r.z * inv, a.out_f32);
        store_out<T>(a.out, o + 3, r.w * inv, a.out_f32);
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

bool quant_mma_shape_ok(int dim, int group_size) {
    return (dim == 64 || dim == 128 || dim == 256) && (group_size == 32 || group_size == 64);
}

bool quant_mma_wide(int rep, int dim, int group_size) {
    return rep >= 16 && (dim == 64 || dim == 128) && (group_size == 32 || group_size == 64);
}

int quant_mma_rows(int rep, int dim, int group_size) { return quant_mma_wide(rep, dim, group_size) ? 16 : 4; }

cudaError_t launch_quant_mma(const QuantArgs &a, cudaStream_t s) {
    if (!quant_mma_shape_ok(a.dim, a.G)) return cudaErrorInvalidValue;
    if (quant_mma_wide(a.rep, a.dim, a.G)) {
        if (a.bits == 4) return launch_quant_mma16_b4(a, s);
        if (a.bits == 8) return launch_quant_mma16_b8(a, s);
        return cudaErrorInvalidValue;
    }
    if (a.bits == 4) return launch_quant_mma_b4(a, s);
    if (a.bits == 8) return launch_quant_mma_b8(a, s);
    return cudaErrorInvalidValue;
}

int quant_mma_ctas_per_sm(int bits, int dim, int ng, int rep) {
    if (ng <= 0 || !quant_mma_shape_ok(dim, dim / ng)) return 0;
    if (quant_mma_wide(rep, dim, dim / ng)) {
        if (bits == 4) return quant_mma16_ctas_per_sm_b4(dim, ng);
        if (bits == 8) return quant_mma16_ctas_per_sm_b8(dim, ng);
        return 0;
    }
    int n = 0;
    if (bits == 4) n = quant_mma_ctas_per_sm_b4(dim, ng);
    if (bits == 8) n = quant_mma_ctas_per_sm_b8(dim, ng);
    // the two-warp form (more than 32 packed words per token) measured fastest
    // with its splits sized for 6 CTAs per SM (8-bit workload: 47.0 us at 6,
    // 48.7 at 7)
    if (dim * bits / 32 > 32 && n > kQmmaTwoWarpCtasPerSm) n = kQmmaTwoWarpCtasPerSm;
    return n;
}

int quant_tc_ctas_per_sm(int bits, int rp, size_t smem) {
    if (bits == 4) return quant_tc_ctas_per_sm_b4(rp, smem);
    if (bits == 8) return quant_tc_ctas_per_sm_b8(rp, smem);
    return 0;
}

cudaError_t launch_quant_tc(const QuantArgs &a, size_t smem, cudaStream_t s) {
    if (a.bits == 4) return launch_quant_tc_b4(a, smem, s);
    if (a.bits == 8) return launch_quant_tc_b8(a, smem, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_quant_merge(const QuantArgs &a, cudaStream_t s) {
    cudaError_t e = a.t_is_bf16 ? launch_pdl(quant_merge_kernel<__nv_bfloat16>, dim3(a.rows), dim3(kMergeThreads), 0, s, a)
                                : launch_pdl(quant_merge_kernel<__half>, dim3(a.rows), dim3(kMergeThreads), 0, s, a);
    count_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace ta
