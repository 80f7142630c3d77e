// Attention over an affine-quantized K/V cache (CUDA cores), split over tokens.
//
// Semantics follow metaltile-std flash_quantized_sdpa.rs (base, bool-mask and
// float-mask kernels): the query is multiplied by `scale` once; K and V are
// dequantized inline (element d = scale[d / G] * code + bias[d / G], code at
// bits (d % pf) * bits of word d / pf); a token is used when it lies in the
// sliding window and its bool-mask slot is non-zero; the float mask is added
// to the logit; the sink is a virtual key with logit sinks[q % nQ] and value
// 0; out = o / l when l > 0, else o.  Applying both masks in one pass is the
// "chained" composition the module doc describes.
//
// GB300 layout (not the pages' one-simdgroup-per-query serial token loop): one
// CTA per (KV row, token split) serving all `repeat` query rows of that KV
// row, so each packed K/V word is read from HBM once per KV row.  Each warp
// walks 32-token chunks: lane = token for the logits (the whole token's codes
// dequantized once, dotted with every query row), then lane = packed word for
// O += p * v.  Online-softmax state is kept per warp, combined across the
// CTA's warps, and either normalized in place (one split) or written as a
// partial (S, M, O) for the merge kernel, which also adds the sink term once.
#include <type_traits>

#include "ta_internal.cuh"

namespace ta {

namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;

template <typename T>
__device__ __forceinline__ float ld_t(const void *p, size_t i) {
    return to_f32(reinterpret_cast<const T *>(p)[i]);
}

template <typename T>
__device__ __forceinline__ void st_out(void *p, size_t i, float x, int out_f32) {
    if (out_f32) reinterpret_cast<float *>(p)[i] = x;
    else if constexpr (sizeof(T) == 2) {
        if constexpr (std::is_same<T, __half>::value) reinterpret_cast<__half *>(p)[i] = __float2half_rn(x);
        else reinterpret_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(x);
    }
}

// Exact small-integer to float: OR the code into the mantissa of 2^23 and
// subtract 2^23 (codes < 2^23 are exact).
__device__ __forceinline__ float code_to_f32(uint32_t code) {
    return __uint_as_float(0x4B000000u | code) - 8388608.0f;
}

// Shared memory of one CTA: scale * q as [dim][REP] (all rows of one element
// in one vector load), the per-group sums of scale * q (bias term of the
// factored dequant), per warp a double-buffered [32 tokens][WPT + 4] tile of
// packed K words (padded so per-token 16-byte reads are conflict-free) and the
// chunk's softmax weights, and the cross-warp combine area.
template <int REP>
struct QuantSmem {
    static size_t qv_floats(int dim, int ng) { return (size_t)REP * dim + (size_t)REP * ng; }
    static size_t bytes(int dim, int ng, int wpt) {
        return sizeof(float) * (qv_floats(dim, ng) + kWarps * 32 * REP + (size_t)kWarps * REP * dim +
                                kWarps * REP * 2) +
               sizeof(uint32_t) * (size_t)kWarps * 2 * 32 * (wpt + 4) + 16;
    }
};

__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool pred) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(pred ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int BITS, typename T, int REP, int WPL>
__global__ void __launch_bounds__(kThreads) quant_fma_kernel(const QuantArgs a) {
    constexpr int PF = 32 / BITS;
    constexpr uint32_t CMASK = (1u << BITS) - 1u;
    constexpr int EPL = WPL * PF;               // output elements per lane
    extern __shared__ __align__(16) float qsm[];
    const int dim = a.dim;
    const int WPT = dim / PF;                   // packed words per token (a multiple of 4)
    const int NG = dim / a.G;
    const int WPG = a.G / PF;                   // words per group
    const int WPS = WPT + 4;                    // padded words per staged token
    float *sQ = qsm;                            // [dim][REP], scale * q
    float *sQg = sQ + REP * dim;                // [REP][NG], per-group sum of scale * q
    float *sP = sQg + REP * NG;                 // [warp][token][REP]
    float *sRed = sP + kWarps * 32 * REP;       // [warp][REP][dim]
    float *sMS = sRed + kWarps * REP * dim;     // [warp][REP][2]
    uint32_t *sK = reinterpret_cast<uint32_t *>(
        (reinterpret_cast<uintptr_t>(sMS + kWarps * REP * 2) + 15) & ~static_cast<uintptr_t>(15));

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, kv = blockIdx.y;
    const int q0 = kv * a.rep;
    const int N = a.N;

    for (int idx = tid; idx < REP * dim; idx += kThreads) {
        const int d = idx / REP, rr = idx % REP;
        sQ[idx] = rr < a.rep ? a.scale * ld_t<T>(a.queries, (size_t)(q0 + rr) * dim + d) : 0.0f;
    }
    __syncthreads();
    for (int idx = tid; idx < REP * NG; idx += kThreads) {
        const int rr = idx / NG, g = idx % NG;
        float acc = 0.0f;
        for (int d = g * a.G; d < (g + 1) * a.G; ++d) acc += sQ[d * REP + rr];
        sQg[idx] = acc;
    }
    __syncthreads();

    // PV lane mapping: lane -> (token offset, word slot)
    const int wpt_eff = WPT < 32 ? WPT : 32;
    const int tpi = 32 / wpt_eff;               // tokens per warp iteration
    const int my_to = lane / wpt_eff;
    const int my_slot = lane % wpt_eff;
    const bool pv_lane = my_to < tpi;

    float M[REP], S[REP], O[REP][EPL], OB[REP][WPL];   // OB: per-word bias term sum_t p * b
#pragma unroll
    for (int rr = 0; rr < REP; ++rr) {
        M[rr] = kMInit;
        S[rr] = 0.0f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) O[rr][e] = 0.0f;
#pragma unroll
        for (int u = 0; u < WPL; ++u) OB[rr][u] = 0.0f;
    }

    const int t_begin = a.t_lo + split * a.tps;
    const int t_end = min(N, t_begin + a.tps);
    float *myP = sP + warp * 32 * REP;
    uint32_t *myK = sK + (size_t)warp * 2 * 32 * WPS;
    const uint32_t *kp_row = a.kp + (size_t)kv * N * WPT;

    // stage the packed K words of the warp's chunk starting at c0 into buffer b
    auto stage_k = [&](int c0, int b) {
        uint32_t *dst = myK + b * 32 * WPS;
        const int pieces = 32 * (WPT / 4);
        for (int i = lane; i < pieces; i += 32) {
            const int tk = i / (WPT / 4), j = i % (WPT / 4);
            const bool ok = c0 + tk < t_end;
            cp_async16(dst + tk * WPS + 4 * j, kp_row + (size_t)(ok ? c0 + tk : t_begin) * WPT + 4 * j, ok);
        }
        cp_async_commit();
    };

    int c0 = t_begin + warp * 32;
    int buf = 0;
    if (c0 < t_end) stage_k(c0, 0);
    for (; c0 < t_end; c0 += kWarps * 32, buf ^= 1) {
        const int cn = c0 + kWarps * 32;
        if (cn < t_end) {
            stage_k(cn, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncwarp();
        // ---- logits: lane = token
        const int t = c0 + lane;
        const bool valid = t < t_end;
        bool gate[REP];
        bool any_gate = false;
#pragma unroll
        for (int rr = 0; rr < REP; ++rr) {
            bool g = valid && (rr < a.rep);
            if (g && a.mbool != nullptr) g = __ldg(a.mbool + (size_t)(q0 + rr) * N + t) != 0u;
            gate[rr] = g;
            any_gate |= g;
        }
        float fm[REP];
#pragma unroll
        for (int rr = 0; rr < REP; ++rr)
            fm[rr] = (a.mfloat != nullptr && gate[rr]) ? ld_t<T>(a.mfloat, (size_t)(q0 + rr) * N + t) : 0.0f;
        float logit[REP];
#pragma unroll
        for (int rr = 0; rr < REP; ++rr) logit[rr] = -INFINITY;
        if (__any_sync(0xffffffffu, any_gate)) {
            float acc[REP];
#pragma unroll
            for (int rr = 0; rr < REP; ++rr) acc[rr] = 0.0f;
            if (any_gate) {
                const size_t tok = (size_t)kv * N + t;
                const uint32_t *kw = myK + buf * 32 * WPS + lane * WPS;
                for (int g = 0; g < NG; ++g) {
                    // q . k over group g = s * sum(q_d * code_d) + b * sum(q_d)
                    float part[REP];
#pragma unroll
                    for (int rr = 0; rr < REP; ++rr) part[rr] = 0.0f;
                    for (int wi = g * WPG; wi < (g + 1) * WPG; wi += 4) {
                        const uint4 w4 = *reinterpret_cast<const uint4 *>(kw + wi);
                        const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
#pragma unroll
                            for (int e = 0; e < PF; ++e) {
                                const float cf = code_to_f32((ws[x] >> (e * BITS)) & CMASK);
                                const float *qd = sQ + ((wi + x) * PF + e) * REP;
#pragma unroll
                                for (int rr = 0; rr < REP; ++rr) part[rr] = fmaf(qd[rr], cf, part[rr]);
                            }
                        }
                    }
                    const float sc = ld_t<T>(a.ks, tok * NG + g);
                    const float bi = ld_t<T>(a.kb, tok * NG + g);
#pragma unroll
                    for (int rr = 0; rr < REP; ++rr)
                        acc[rr] = fmaf(sc, part[rr], fmaf(bi, sQg[rr * NG + g], acc[rr]));
                }
            }
#pragma unroll
            for (int rr = 0; rr < REP; ++rr) logit[rr] = gate[rr] ? acc[rr] + fm[rr] : -INFINITY;
        }
        // ---- online softmax over the 32 tokens, per row
#pragma unroll
        for (int rr = 0; rr < REP; ++rr) {
            const float cm = warp_max(logit[rr]);
            float p = 0.0f;
            if (cm != -INFINITY) {
                const float m_new = fmaxf(M[rr], cm);
                const float alpha = expf(M[rr] - m_new);
                p = expf(logit[rr] - m_new);
                S[rr] = S[rr] * alpha + warp_sum(p);
                M[rr] = m_new;
#pragma unroll
                for (int e = 0; e < EPL; ++e) O[rr][e] *= alpha;
#pragma unroll
                for (int u = 0; u < WPL; ++u) OB[rr][u] *= alpha;
            }
            myP[lane * REP + rr] = p;
        }
        __syncwarp();
        // ---- O += p * v = (p * s) * code + p * b: lane = packed word
        if (pv_lane) {
#pragma unroll 2
            for (int tt = 0; tt < 32; tt += tpi) {
                const int to = tt + my_to;
                const int tk = c0 + to;
                if (to >= 32 || tk >= t_end) break;
                float pw[REP];
                bool any_p = false;
#pragma unroll
                for (int rr = 0; rr < REP; ++rr) { pw[rr] = myP[to * REP + rr]; any_p |= pw[rr] != 0.0f; }
                if (!any_p) continue;
                const size_t tok = (size_t)kv * N + tk;
                uint32_t wv[WPL];
                float sv[WPL], bv[WPL];
#pragma unroll
                for (int u = 0; u < WPL; ++u) {
                    const int wi = my_slot + 32 * u;
                    const bool in = wi < WPT;
                    wv[u] = in ? __ldg(a.vp + tok * WPT + wi) : 0u;
                    sv[u] = in ? ld_t<T>(a.vs, tok * NG + wi / WPG) : 0.0f;
                    bv[u] = in ? ld_t<T>(a.vb, tok * NG + wi / WPG) : 0.0f;
                }
#pragma unroll
                for (int u = 0; u < WPL; ++u) {
                    float ps[REP];
#pragma unroll
                    for (int rr = 0; rr < REP; ++rr) {
                        ps[rr] = pw[rr] * sv[u];
                        OB[rr][u] = fmaf(pw[rr], bv[u], OB[rr][u]);
                    }
#pragma unroll
                    for (int e = 0; e < PF; ++e) {
                        const float cf = code_to_f32((wv[u] >> (e * BITS)) & CMASK);
#pragma unroll
                        for (int rr = 0; rr < REP; ++rr) O[rr][u * PF + e] = fmaf(ps[rr], cf, O[rr][u * PF + e]);
                    }
                }
            }
        }
        __syncwarp();
    }
#pragma unroll
    for (int rr = 0; rr < REP; ++rr)
#pragma unroll
        for (int u = 0; u < WPL; ++u)
#pragma unroll
            for (int e = 0; e < PF; ++e) O[rr][u * PF + e] += OB[rr][u];

    // ---- lanes sharing a word slot hold the same state: sum them
    for (int k = 1; k < tpi; ++k) {
#pragma unroll
        for (int rr = 0; rr < REP; ++rr)
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                const int src = lane + k * wpt_eff;
                const float x = __shfl_sync(0xffffffffu, O[rr][e], src < 32 ? src : lane);
                if (lane < wpt_eff) O[rr][e] += x;
            }
    }
    // ---- combine the CTA's warps
    if (lane == 0) {
#pragma unroll
        for (int rr = 0; rr < REP; ++rr) {
            sMS[(warp * REP + rr) * 2 + 0] = M[rr];
            sMS[(warp * REP + rr) * 2 + 1] = S[rr];
        }
    }
    __syncthreads();
    float wscale[REP];
#pragma unroll
    for (int rr = 0; rr < REP; ++rr) {
        float mstar = -FLT_MAX;
        for (int w = 0; w < kWarps; ++w) mstar = fmaxf(mstar, sMS[(w * REP + rr) * 2]);
        wscale[rr] = expf(M[rr] - mstar);
    }
    if (lane < wpt_eff) {
#pragma unroll
        for (int rr = 0; rr < REP; ++rr)
#pragma unroll
            for (int u = 0; u < WPL; ++u) {
                const int wi = my_slot + 32 * u;
                if (wi >= WPT) break;
#pragma unroll
                for (int e = 0; e < PF; ++e)
                    sRed[((size_t)warp * REP + rr) * dim + wi * PF + e] = O[rr][u * PF + e] * wscale[rr];
            }
    }
    __syncthreads();
    for (int idx = tid; idx < a.rep * dim; idx += kThreads) {
        const int rr = idx / dim, d = idx % dim;
        float mstar = -FLT_MAX, sstar = 0.0f, o = 0.0f;
        for (int w = 0; w < kWarps; ++w) mstar = fmaxf(mstar, sMS[(w * REP + rr) * 2]);
        for (int w = 0; w < kWarps; ++w) {
            sstar += sMS[(w * REP + rr) * 2 + 1] * expf(sMS[(w * REP + rr) * 2] - mstar);
            o += sRed[((size_t)w * REP + rr) * dim + d];
        }
        const int q = q0 + rr;
        if (a.nwg == 1) {
            float mf = mstar, sf = sstar, of = o;
            if (a.has_sinks) {
                const float sink = __ldg(a.sinks + (q % a.nQ));
                mf = fmaxf(mstar, sink);
                const float c = expf(mstar - mf);
                sf = sstar * c + expf(sink - mf);
                of = o * c;
            }
            st_out<T>(a.out, (size_t)q * dim + d, sf > 0.0f ? of / sf : of, a.out_f32);
        } else {
            a.part_o[((size_t)split * a.rows + q) * dim + d] = o;
            if (d == 0) {
                a.part_ml[((size_t)split * a.rows + q) * 2 + 0] = sstar;
                a.part_ml[((size_t)split * a.rows + q) * 2 + 1] = mstar;
            }
        }
    }
}

// Merge of the token-split partials, plus the sink term, into out (T or f32).
template <typename T>
__global__ void __launch_bounds__(128) quant_merge_kernel(const QuantArgs a) {
    const int q = blockIdx.x;
    float mstar = -FLT_MAX;
    for (int w = 0; w < a.nwg; ++w) mstar = fmaxf(mstar, __ldg(a.part_ml + ((size_t)w * a.rows + q) * 2 + 1));
    float sink = 0.0f;
    if (a.has_sinks) {
        sink = __ldg(a.sinks + (q % a.nQ));
        mstar = fmaxf(mstar, sink);
    }
    float sstar = a.has_sinks ? expf(sink - mstar) : 0.0f;
    for (int w = 0; w < a.nwg; ++w) {
        const float sw = __ldg(a.part_ml + ((size_t)w * a.rows + q) * 2 + 0);
        const float mw = __ldg(a.part_ml + ((size_t)w * a.rows + q) * 2 + 1);
        sstar += sw * expf(mw - mstar);
    }
    for (int d = threadIdx.x; d < a.dim; d += blockDim.x) {
        float o = 0.0f;
        for (int w = 0; w < a.nwg; ++w) {
            const float mw = __ldg(a.part_ml + ((size_t)w * a.rows + q) * 2 + 1);
            o += __ldg(a.part_o + ((size_t)w * a.rows + q) * a.dim + d) * expf(mw - mstar);
        }
        st_out<T>(a.out, (size_t)q * a.dim + d, sstar > 0.0f ? o / sstar : o, a.out_f32);
    }
}

template <int BITS, typename T, int REP, int WPL>
cudaError_t launch_q(const QuantArgs &a, cudaStream_t s) {
    auto kern = quant_fma_kernel<BITS, T, REP, WPL>;
    const size_t smem = QuantSmem<REP>::bytes(a.dim, a.dim / a.G, a.dim * BITS / 32);
    static unsigned long long done = 0;
    cudaError_t e = set_smem_limit_once(kern, smem, &done);
    if (e != cudaSuccess) return e;
    dim3 grid(a.nwg, a.kv_rows);
    kern<<<grid, kThreads, smem, s>>>(a);
    count_launch();
    return cudaGetLastError();
}

template <int BITS, typename T, int REP>
cudaError_t launch_q_wpl(const QuantArgs &a, cudaStream_t s) {
    const int wpt = a.dim * BITS / 32;
    const int wpl = (wpt + 31) / 32;
    if (wpl <= 1) return launch_q<BITS, T, REP, 1>(a, s);
    if (wpl <= 2) return launch_q<BITS, T, REP, 2>(a, s);
    if (wpl <= 4) return launch_q<BITS, T, REP, 4>(a, s);
    return cudaErrorInvalidValue;
}

template <int BITS, typename T>
cudaError_t launch_q_rep(const QuantArgs &a, cudaStream_t s) {
    if (a.rep <= 4) return launch_q_wpl<BITS, T, 4>(a, s);
    if (a.rep <= 8) return launch_q_wpl<BITS, T, 8>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_quant_fma(const QuantArgs &a, cudaStream_t s) {
    if (a.bits == 4) return a.t_is_bf16 ? launch_q_rep<4, __nv_bfloat16>(a, s) : launch_q_rep<4, __half>(a, s);
    if (a.bits == 8) return a.t_is_bf16 ? launch_q_rep<8, __nv_bfloat16>(a, s) : launch_q_rep<8, __half>(a, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_quant_merge(const QuantArgs &a, cudaStream_t s) {
    dim3 grid(a.rows);
    if (a.t_is_bf16) quant_merge_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(a);
    else quant_merge_kernel<__half><<<grid, 128, 0, s>>>(a);
    count_launch();
    return cudaGetLastError();
}

}  // namespace ta
