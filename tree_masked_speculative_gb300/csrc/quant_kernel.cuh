// Attention over an affine-quantized K/V cache on the CUDA cores (one warp
// per CTA).  Included by quant_b4.cu and quant_b8.cu, which instantiate it.
//
// What it computes follows metaltile-std flash_quantized_sdpa.rs (base,
// bool-mask and float-mask kernels): q is multiplied by `scale` before the dot;
// K and V element d of a token is scale[d / G] * code_d + bias[d / G], code_d
// at bits (d % pf) * bits of word d / pf; a token takes part when it lies in
// the sliding window and its bool-mask slot is non-zero; the float mask is
// added to the logit; the sink is a virtual key with logit sinks[q % nQ] and
// value 0 (added by the finalisation or the merge); out = o / l, or o when
// l = 0.  Both masks applied in one pass is the chained composition the
// module doc describes.
//
// GB300 design (not the pages' one-simdgroup-per-query token loop):
//  * one warp = one CTA owns a (KV row, row group of 4 query rows, token
//    split); the split count fills every SM's resident-warp slots in one wave;
//  * every chunk (32 tokens, or 16 when a token has more than 32 packed
//    words) is staged in shared memory in two groups (K words + scales +
//    masks, then V words), each double-buffered and issued two chunks ahead:
//    the K and V tiles by TMA bulk copies, the small scale and mask runs by
//    per-lane cp.async, all completing on mbarriers;
//  * scores: each lane keeps scale * log2(e) * q for 16 dimensions of the 4
//    rows in registers (so no shared-memory broadcast of q per dimension),
//    decodes its part of each token with byte permutes, scales the codes with
//    one packed FMA (s * (2^23 + c) - 2^23 * s = s * c) and accumulates with
//    packed f32x2 FMAs; the per-token partial sums of the lanes are combined
//    by a transposed butterfly (reduce-scatter), which leaves each lane one
//    (token, row) score per batch of passes; the bias term sum_g b_g * sum_{d in g} q_d
//    is added once per (token, row) after the reduction;
//  * online softmax in log2 units per row; P is kept in shared memory;
//  * values: lane = packed-word slot; O += p * (s * c) with the same decode
//    and packed FMAs, and the bias part sum_t p_t * b_t is accumulated per
//    (row, group) once per chunk.
#pragma once

#include <type_traits>

#include "sm100_ptx.cuh"
#include "ta_internal.cuh"

namespace ta {
namespace quant {

using namespace ta::sm100;

constexpr int REP = kQuantRowsPerCta;   // query rows of one row group
constexpr int DPL = 16;                 // score pass: dimensions per lane (q regs = DPL * REP)
constexpr float kSlack = 8.0f;              // lazy-max slack (log2 units)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTwo23 = 8388608.0f;   // 2^23: the float whose low mantissa bits hold a code

template <int BITS, int DIMC>
struct Shape {
    static constexpr int CH = DIMC * BITS / 32 <= 32 ? 32 : 16;   // tokens per chunk
    static constexpr int NB = CH * REP / 32;               // score slots (token, row) per lane
    static constexpr int PF = 32 / BITS;                   // codes per packed word
    static constexpr int LPT = DIMC / DPL;                 // score lanes per token (4..32)
    static constexpr int TPP = 32 / LPT;                   // tokens per score pass
    static constexpr int B = LPT / REP;                    // score passes per reduction batch
    static constexpr int WPQ = DPL / PF;                   // words per lane per token (scores)
    static constexpr int WPTC = DIMC * BITS / 32;          // words per token at capacity
    static constexpr int WPL = WPTC >= 32 ? WPTC / 32 : 1; // words per lane (values)
    static constexpr int LPV = WPTC / WPL;                 // value lanes per token
    static constexpr int TPV = 32 / LPV;                   // tokens per value pass
    static constexpr int EPL = WPL * PF;                   // output dimensions per lane
    static_assert(LPT >= REP && LPT <= 32, "score lanes per token");
    static_assert(B * REP == LPT, "one reduced score per lane per batch");
    static_assert(REP == 4, "the value pass reads the weights of four rows");
    static_assert(NB * B * TPP == CH && CH % TPV == 0, "chunk tiling");
    static_assert(CH == 32 || CH == 16, "chunk length");
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// cp.async of 16 bytes (zero-filled beyond src_bytes) and of 4 bytes; the
// thread's prior cp.async copies arrive on an mbarrier once they have landed
// (.noinc: the barrier's expected count includes these arrivals).
__device__ __forceinline__ void cp16(void *dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp4(void *dst, const void *src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Bounded wait of every lane on an mbarrier phase; the result is uniform.
__device__ __forceinline__ bool wait_warp(uint64_t *bar, uint32_t parity, uint32_t polls = kQuantWaitPolls) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, polls));
}

template <typename T>
__device__ __forceinline__ float t2f(uint16_t bits) {
    if constexpr (std::is_same<T, __nv_bfloat16>::value) return __uint_as_float(static_cast<uint32_t>(bits) << 16);
    else return __half2float(__ushort_as_half(bits));
}

template <typename T>
__device__ __forceinline__ void st_out(void *p, size_t i, float x, int out_f32) {
    if (out_f32) reinterpret_cast<float *>(p)[i] = x;
    else if constexpr (std::is_same<T, __half>::value) reinterpret_cast<__half *>(p)[i] = __float2half_rn(x);
    else reinterpret_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(x);
}

// Codes (2k, 2k+1) of a packed word as the floats {2^23 + c0, 2^23 + c1}: the
// code byte is permuted into the low mantissa byte under the exponent of 2^23.
template <int BITS>
struct Codes;
template <>
struct Codes<8> {
    uint32_t w;
    __device__ __forceinline__ explicit Codes(uint32_t word) : w(word) {}
    __device__ __forceinline__ float2 pair(int k) const {
        return make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u | (2 * k))),
                           __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u | (2 * k + 1))));
    }
};
template <>
struct Codes<4> {
    uint32_t lo, hi;   // even / odd nibbles, one per byte
    __device__ __forceinline__ explicit Codes(uint32_t w) : lo(w & 0x0F0F0F0Fu), hi((w >> 4) & 0x0F0F0F0Fu) {}
    __device__ __forceinline__ float2 pair(int k) const {
        return make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7440u | k)),
                           __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7440u | k)));
    }
};

// Reduce-scatter over groups of N lanes (xor 1 .. N/2): on return lane l holds
// the sum over its group of value index (l % N).
template <int N>
__device__ __forceinline__ float reduce_scatter(float (&v)[N], int lane) {
#pragma unroll
    for (int s = 0; (1 << s) < N; ++s) {
        const int m = 1 << s;
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int k = 0; k < (N >> s) / 2; ++k) {
            const float send = upper ? v[2 * k] : v[2 * k + 1];
            const float keep = upper ? v[2 * k + 1] : v[2 * k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
    }
    return v[0];
}

template <typename T, int WPL>
__device__ __forceinline__ void load_words(const uint32_t *p, uint32_t (&w)[WPL]) {
    if constexpr (WPL == 4) {
        const uint4 x = *reinterpret_cast<const uint4 *>(p);
        w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
    } else if constexpr (WPL == 2) {
        const uint2 x = *reinterpret_cast<const uint2 *>(p);
        w[0] = x.x; w[1] = x.y;
    } else {
#pragma unroll
        for (int u = 0; u < WPL; ++u) w[u] = p[u];
    }
}

// GC > 0: exact-shape instance (dim == DIMC, group size GC, both compile-time
// so that shared-memory addressing folds into immediates); GC == 0: any
// dim <= DIMC and group size, read at run time.
// Chunk staging shared by the quantized-KV kernels (one warp stages its own
// chunks).  Group A of chunk c into stage b: lane 0 copies the K tile with one
// bulk copy (mbarrier transaction bytes); the scale / bias runs and mask rows
// are copied by all lanes with 16- or 4-byte cp.async that arrive on the same
// mbarrier (count 1 + 32); tail chunks and unaligned rows are filled with
// plain loads (zero beyond N).  Group B: lane 0 copies the V tile.
template <int CH>
struct QuantStager {
    const QuantArgs &a;
    const QuantLayout &L;
    unsigned char *smem;
    uint64_t *bars;   // A stages 0 .. ns-1, then B stages 0 .. ns-1
    int WPT, NG, kv, q0, nrow, lane, ns;
    bool with_k;      // issue_a also copies the K tile (else another warp does)

    __device__ __forceinline__ void issue_a(int c, int b) const {
        const int N = a.N;
        unsigned char *st = smem + L.a0 + b * L.a_stage;
        const int t0 = c * CH, tval = min(CH, N - t0);
        const bool full = tval == CH;
        const size_t tok0 = static_cast<size_t>(kv) * N + t0;
        if (lane == 0 && with_k) {
            const uint32_t kbytes = static_cast<uint32_t>(tval * WPT * 4);
            mbar_arrive_expect_tx(&bars[b], kbytes);
            bulk_load(st + L.k, a.kp + tok0 * WPT, kbytes, &bars[b]);
        }
        // scale / bias runs: [4 arrays][CH * NG] T
        {
            const int per = CH * NG;   // elements per array
            if (a.al_sb && full) {
                const int pieces = per / 8;
                for (int i = lane; i < 4 * pieces; i += 32) {
                    const int arr = i / pieces, pc = i % pieces;
                    const void *base = arr == 0 ? a.ks : arr == 1 ? a.kb : arr == 2 ? a.vs : a.vb;
                    const int off = arr == 0 ? L.ks : arr == 1 ? L.kb : arr == 2 ? L.vs : L.vb;
                    cp16(st + off + 16 * pc, static_cast<const uint16_t *>(base) + tok0 * NG + 8 * pc, 16);
                }
            } else {
                const int valid = tval * NG;
                for (int i = lane; i < 4 * per; i += 32) {
                    const int arr = i / per, e = i % per;
                    const void *base = arr == 0 ? a.ks : arr == 1 ? a.kb : arr == 2 ? a.vs : a.vb;
                    const int off = arr == 0 ? L.ks : arr == 1 ? L.kb : arr == 2 ? L.vs : L.vb;
                    reinterpret_cast<uint16_t *>(st + off)[e] =
                        e < valid ? static_cast<const uint16_t *>(base)[tok0 * NG + e] : static_cast<uint16_t>(0);
                }
            }
        }
        // bool-mask rows [REP][CH] u32 (rows beyond nrow are never read)
        if (a.mbool != nullptr) {
            uint32_t *dst = reinterpret_cast<uint32_t *>(st + L.mb);
            if (a.al_mb && full) {
                for (int i = lane; i < nrow * CH / 4; i += 32) {
                    const int r = i / (CH / 4), pc = i % (CH / 4);
                    cp16(dst + r * CH + 4 * pc, a.mbool + static_cast<size_t>(q0 + r) * N + t0 + 4 * pc, 16);
                }
            } else {
                for (int i = lane; i < nrow * CH; i += 32) {
                    const int r = i / CH, t = i % CH;
                    const uint32_t *src = a.mbool + static_cast<size_t>(q0 + r) * N + t0;
                    cp4(dst + i, t < tval ? src + t : src, t < tval ? 4 : 0);
                }
            }
        }
        // float-mask rows [REP][CH] T
        if (a.mfloat != nullptr) {
            const uint16_t *mf = static_cast<const uint16_t *>(a.mfloat);
            uint16_t *dst = reinterpret_cast<uint16_t *>(st + L.mf);
            if (a.al_mf && full) {
                for (int i = lane; i < nrow * CH / 8; i += 32) {
                    const int r = i / (CH / 8), pc = i % (CH / 8);
                    cp16(dst + r * CH + 8 * pc, mf + static_cast<size_t>(q0 + r) * N + t0 + 8 * pc, 16);
                }
            } else {
                for (int i = lane; i < nrow * CH; i += 32) {
                    const int r = i / CH, t = i % CH;
                    dst[i] = t < tval ? mf[static_cast<size_t>(q0 + r) * N + t0 + t] : static_cast<uint16_t>(0);
                }
            }
        }
        cp_arrive_noinc(&bars[b]);
    }
    __device__ __forceinline__ void issue_b(int c, int b) const {
        const int N = a.N;
        if (lane == 0) {
            const int t0 = c * CH, tval = min(CH, N - t0);
            const uint32_t bytes = static_cast<uint32_t>(tval * WPT * 4);
            mbar_arrive_expect_tx(&bars[ns + b], bytes);
            bulk_load(smem + L.v0 + b * L.v_stage, a.vp + (static_cast<size_t>(kv) * N + t0) * WPT, bytes,
                      &bars[ns + b]);
        }
    }
};

template <int BITS, typename T, int DIMC, int GC>
__global__ void __launch_bounds__(32, (DIMC >= 512 ? 8 : 12)) quant_kernel(const QuantArgs a) {
    using S = Shape<BITS, DIMC>;
    constexpr int CH = S::CH, NB = S::NB;
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x;
    const int rg = blockIdx.x % a.n_rg, split = blockIdx.x / a.n_rg, kv = blockIdx.y;
    const int q0 = kv * a.rep + rg * REP;
    const int nrow = min(REP, a.rep - rg * REP);
    const int N = a.N;
    const int WPT = GC > 0 ? DIMC * BITS / 32 : a.wpt;
    const int NG = GC > 0 ? DIMC / (GC > 0 ? GC : 1) : a.ng;
    const int G = GC > 0 ? GC : a.G;
    const int dim = GC > 0 ? DIMC : a.dim;
    const QuantLayout L = quant_layout(WPT, NG, CH);
    float4 *sKS4 = reinterpret_cast<float4 *>(smem + L.ks4);   // {s, s, -2^23 s, -2^23 s}
    float4 *sVS4 = reinterpret_cast<float4 *>(smem + L.vs4);
    float2 *sP2 = reinterpret_cast<float2 *>(smem + L.p2);     // [token][row] {p, p}
    float *sOBl = reinterpret_cast<float *>(smem + L.ob);      // [group][lane] sum_t p * b (lane's slots)
    float *sQS = reinterpret_cast<float *>(smem + L.qs);       // [row][group] sum_{d in g} q'
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);   // A stage 0/1, B stage 0/1

    const int c_begin = a.c_lo + static_cast<int>((static_cast<long long>(split) * a.nch) / a.nwg);
    const int c_end = a.c_lo + static_cast<int>((static_cast<long long>(split + 1) * a.nch) / a.nwg);
    const int nc = c_end - c_begin;

    // score-pass roles: lane = (token in pass tp, dimension slice j)
    const int tp = lane / S::LPT, j = lane % S::LPT;
    const int d0 = j * DPL;
    const bool qk_live = d0 < dim;
    const int g_qk = qk_live ? d0 / G : 0;
    const int r_l = j % REP;   // row of the lane's reduced scores
    // draft tree over the last tree_ql tokens: the ancestor bitset of the lane's
    // row's node (lane i < tree_ql builds node i's, the row's node takes it)
    const int tree_lo = N - a.tree_ql;
    uint32_t tree_bits = 0u;
    if (a.tree_ql > 0) {
        const uint32_t mine =
            quant_tree_ancestors(lane < a.tree_ql ? __ldg(a.tree_parents + lane) : -1, a.tree_ql);
        tree_bits = __shfl_sync(0xffffffffu, mine, (q0 + r_l) % a.tree_ql);
    }
    const int pb_l = j / REP;  // pass (within a batch) of the lane's reduced scores
    // value-pass roles: lane = (token in pass tv, word slot wl)
    const int tv = lane / S::LPV, wl = lane % S::LPV;
    const bool pv_live = wl * S::WPL < WPT;
    const int g_v = pv_live ? (wl * S::WPL * S::PF) / G : 0;

    if (lane == 0) {
        mbar_init(&bars[0], 33);   // group A: lane 0's expect-tx arrive + one cp.async arrive per lane
        mbar_init(&bars[1], 33);
        mbar_init(&bars[2], 1);    // group B: lane 0's expect-tx arrive
        mbar_init(&bars[3], 1);
        fence_mbar_init();
    }
    __syncwarp();

    const QuantStager<CH> stg{a, L, smem, bars, WPT, NG, kv, q0, nrow, lane, 2, true};
    auto issue_a = [&](int c, int b) { stg.issue_a(c, b); };
    auto issue_b = [&](int c, int b) { stg.issue_b(c, b); };
    int a_issued = 0, b_issued = 0, a_done = 0, b_done = 0;
    for (; a_issued < 2 && a_issued < nc; ++a_issued) issue_a(c_begin + a_issued, a_issued & 1);
    for (; b_issued < 2 && b_issued < nc; ++b_issued) issue_b(c_begin + b_issued, b_issued & 1);

    // q' = scale * log2(e) * q for the lane's 16 dimensions of every row
    const float qscale = a.scale * kLog2e;
    float2 q2[REP][DPL / 2];
    {
        const uint16_t *qg = reinterpret_cast<const uint16_t *>(a.queries);
#pragma unroll
        for (int r = 0; r < REP; ++r)
#pragma unroll
            for (int k = 0; k < DPL / 2; ++k) {
                float2 x = make_float2(0.0f, 0.0f);
                if (qk_live && r < nrow) {
                    const size_t i = static_cast<size_t>(q0 + r) * dim + d0 + 2 * k;
                    x = make_float2(qscale * t2f<T>(qg[i]), qscale * t2f<T>(qg[i + 1]));
                }
                q2[r][k] = x;
            }
    }
    // per-(row, group) sums of q' (bias term), via the lanes' partial sums
    {
        float *sQP = reinterpret_cast<float *>(sP2);   // [row][LPT], free until the first chunk
        if (tp == 0) {
#pragma unroll
            for (int r = 0; r < REP; ++r) {
                float s = 0.0f;
#pragma unroll
                for (int k = 0; k < DPL / 2; ++k) s += q2[r][k].x + q2[r][k].y;
                sQP[r * S::LPT + j] = s;
            }
        }
        __syncwarp();
        const int lpg = G / DPL;   // lanes per group
        for (int idx = lane; idx < REP * NG; idx += 32) {
            const int r = idx / NG, g = idx % NG;
            float s = 0.0f;
            for (int jj = g * lpg; jj < (g + 1) * lpg; ++jj) s += sQP[r * S::LPT + jj];
            sQS[idx] = s;
        }
        for (int idx = lane; idx < 32 * NG; idx += 32) sOBl[idx] = 0.0f;
        __syncwarp();
    }

    float M = -INFINITY, Ssum = 0.0f;   // online-softmax state of row r_l (log2 units)
    float2 O2[REP][S::EPL / 2];
#pragma unroll
    for (int r = 0; r < REP; ++r)
#pragma unroll
        for (int k = 0; k < S::EPL / 2; ++k) O2[r][k] = make_float2(0.0f, 0.0f);

    bool ok = true;
    for (int i = 0; i < nc; ++i) {
        const int c = c_begin + i, b = i & 1;
        const uint32_t par = static_cast<uint32_t>(i >> 1) & 1u;
        // group A of chunk c (the first wait's bound is a parameter: a test
        // makes it time out to exercise this failure path)
        if (!wait_warp(&bars[b], par, i == 0 ? a.first_wait_polls : kQuantWaitPolls)) { ok = false; break; }
        ++a_done;
        __syncwarp();
        const unsigned char *st = smem + L.a0 + b * L.a_stage;
        const uint32_t *sK = reinterpret_cast<const uint32_t *>(st + L.k);
        const uint16_t *sKs = reinterpret_cast<const uint16_t *>(st + L.ks);
        const uint16_t *sKb = reinterpret_cast<const uint16_t *>(st + L.kb);
        const uint16_t *sVs = reinterpret_cast<const uint16_t *>(st + L.vs);
        const uint16_t *sVb = reinterpret_cast<const uint16_t *>(st + L.vb);
        const uint32_t *sMb = reinterpret_cast<const uint32_t *>(st + L.mb);
        const uint16_t *sMf = reinterpret_cast<const uint16_t *>(st + L.mf);
        const uint32_t *sV = reinterpret_cast<const uint32_t *>(smem + L.v0 + b * L.v_stage);
        const int t0 = c * CH;
        for (int idx = lane; idx < CH * NG; idx += 32) {
            const float s = t2f<T>(sKs[idx]);
            sKS4[idx] = make_float4(s, s, -kTwo23 * s, -kTwo23 * s);
            const float sv = t2f<T>(sVs[idx]);
            sVS4[idx] = make_float4(sv, sv, -kTwo23 * sv, -kTwo23 * sv);
        }
        // gates of the lane's (token, row) score slots
        bool live[NB];
        int tk[NB];
        bool any = false;
#pragma unroll
        for (int bb = 0; bb < NB; ++bb) {
            tk[bb] = (bb * S::B + pb_l) * S::TPP + tp;
            const int t = t0 + tk[bb];
            bool g = r_l < nrow && t >= a.t_lo && t < N;
            if (g && a.mbool != nullptr) g = sMb[r_l * CH + tk[bb]] != 0u;
            if (g && a.tree_ql > 0 && t >= tree_lo) g = (tree_bits >> (t - tree_lo)) & 1u;
            live[bb] = g;
            any |= g;
        }
        __syncwarp();
        const bool chunk_live = __any_sync(0xffffffffu, any);

        float lg[NB];
#pragma unroll
        for (int bb = 0; bb < NB; ++bb) lg[bb] = -INFINITY;
        if (chunk_live) {
            // ---- scores: partial dot products, reduce-scattered over the token's lanes
#pragma unroll
            for (int bb = 0; bb < NB; ++bb) {
                float v[S::B * REP];
#pragma unroll
                for (int pb = 0; pb < S::B; ++pb) {
                    const int t = (bb * S::B + pb) * S::TPP + tp;
                    float2 acc[REP];
#pragma unroll
                    for (int r = 0; r < REP; ++r) acc[r] = make_float2(0.0f, 0.0f);
                    if (qk_live) {
                        uint32_t w[S::WPQ];
                        load_words<T, S::WPQ>(sK + t * WPT + d0 / S::PF, w);
                        const float4 sm = sKS4[t * NG + g_qk];
                        const float2 s2 = make_float2(sm.x, sm.y), m2 = make_float2(sm.z, sm.w);
#pragma unroll
                        for (int u = 0; u < S::WPQ; ++u) {
                            const Codes<BITS> cd(w[u]);
#pragma unroll
                            for (int k = 0; k < S::PF / 2; ++k) {
                                const float2 sc = __ffma2_rn(cd.pair(k), s2, m2);   // s * code, rounded once
#pragma unroll
                                for (int r = 0; r < REP; ++r)
                                    acc[r] = __ffma2_rn(q2[r][u * (S::PF / 2) + k], sc, acc[r]);
                            }
                        }
                    }
#pragma unroll
                    for (int r = 0; r < REP; ++r) v[pb * REP + r] = acc[r].x + acc[r].y;
                }
                const float dot = reduce_scatter<S::B * REP>(v, lane);
                if (live[bb]) {
                    // + sum_g b_g * sum_{d in g} q'_d, + log2(e) * float mask
                    float bias = 0.0f;
                    for (int g = 0; g < NG; ++g) bias = fmaf(t2f<T>(sKb[tk[bb] * NG + g]), sQS[r_l * NG + g], bias);
                    float fm = 0.0f;
                    if (a.mfloat != nullptr) fm = kLog2e * t2f<T>(sMf[r_l * CH + tk[bb]]);
                    lg[bb] = dot + bias + fm;
                }
            }
        }

        // ---- online softmax of row r_l (log2 units).  The running max M only
        // moves when a score exceeds it by more than kSlack (then every row is
        // rescaled); otherwise the weights 2^(s - M) <= 2^kSlack are used as
        // they are.  S and the V-bias sums stay per lane until the end.
        bool grow = false;
#pragma unroll
        for (int bb = 0; bb < NB; ++bb) grow |= lg[bb] > M + kSlack;
        if (__any_sync(0xffffffffu, grow)) {
            float cmax = lg[0];
#pragma unroll
            for (int bb = 1; bb < NB; ++bb) cmax = fmaxf(cmax, lg[bb]);
#pragma unroll
            for (int m = REP; m < 32; m <<= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, m));
            const float m_new = fmaxf(M, cmax);
            const float alpha = m_new == M ? 1.0f : ex2(M - m_new);   // 0 while M = -inf
            M = m_new;
            Ssum *= alpha;
            for (int g = 0; g < NG; ++g) sOBl[g * 32 + lane] *= alpha;
            float al[REP];
#pragma unroll
            for (int r = 0; r < REP; ++r) al[r] = __shfl_sync(0xffffffffu, alpha, r);
#pragma unroll
            for (int r = 0; r < REP; ++r)
#pragma unroll
                for (int k = 0; k < S::EPL / 2; ++k) {
                    O2[r][k].x *= al[r];
                    O2[r][k].y *= al[r];
                }
        }
        if (chunk_live) {
            float p[NB];
#pragma unroll
            for (int bb = 0; bb < NB; ++bb) {
                p[bb] = M == -INFINITY ? 0.0f : ex2(lg[bb] - M);
                Ssum += p[bb];
                sP2[tk[bb] * REP + r_l] = make_float2(p[bb], p[bb]);
            }
            // bias part of O: sum_t p_t * b_{t,g}, this lane's slots, per group
            for (int g = 0; g < NG; ++g) {
                float x = sOBl[g * 32 + lane];
#pragma unroll
                for (int bb = 0; bb < NB; ++bb) x = fmaf(p[bb], t2f<T>(sVb[tk[bb] * NG + g]), x);
                sOBl[g * 32 + lane] = x;
            }
        }
        __syncwarp();
        if (a_issued < nc) { issue_a(c_begin + a_issued, a_issued & 1); ++a_issued; }   // stage b is free
        if (!wait_warp(&bars[2 + b], par)) { ok = false; break; }   // group B of chunk c
        ++b_done;
        __syncwarp();

        // ---- values: O += p * (s * code); lane = packed-word slot
        if (chunk_live && pv_live) {
#pragma unroll 4
            for (int ps = 0; ps < CH / S::TPV; ++ps) {
                const int t = ps * S::TPV + tv;
                uint32_t w[S::WPL];
                load_words<T, S::WPL>(sV + t * WPT + wl * S::WPL, w);
                const float4 sm = sVS4[t * NG + g_v];
                const float2 s2 = make_float2(sm.x, sm.y), m2 = make_float2(sm.z, sm.w);
                const float4 pa = *reinterpret_cast<const float4 *>(sP2 + t * REP);
                const float4 pc = *reinterpret_cast<const float4 *>(sP2 + t * REP + 2);
                const float2 pp[REP] = {make_float2(pa.x, pa.y), make_float2(pa.z, pa.w), make_float2(pc.x, pc.y),
                                        make_float2(pc.z, pc.w)};
#pragma unroll
                for (int u = 0; u < S::WPL; ++u) {
                    const Codes<BITS> cd(w[u]);
#pragma unroll
                    for (int k = 0; k < S::PF / 2; ++k) {
                        const float2 sc = __ffma2_rn(cd.pair(k), s2, m2);
#pragma unroll
                        for (int r = 0; r < REP; ++r)
                            O2[r][u * (S::PF / 2) + k] = __ffma2_rn(pp[r], sc, O2[r][u * (S::PF / 2) + k]);
                    }
                }
            }
        }
        __syncwarp();
        if (b_issued < nc) { issue_b(c_begin + b_issued, b_issued & 1); ++b_issued; }
    }
    pdl_launch_dependents();   // the merge may start launching; it waits for this grid to finish
    if (!ok) {
        // a copy never completed: report it, let the issued copies land (bounded) and leave
        if (lane == 0 && a.err != nullptr) atomicOr(a.err, 1);
        for (; a_done < a_issued; ++a_done) wait_warp(&bars[a_done & 1], static_cast<uint32_t>(a_done >> 1) & 1u);
        for (; b_done < b_issued; ++b_done) wait_warp(&bars[2 + (b_done & 1)], static_cast<uint32_t>(b_done >> 1) & 1u);
        return;
    }

    // ---- lanes that share word slots hold sums over different tokens
#pragma unroll
    for (int m = S::LPV; m < 32; m <<= 1)
#pragma unroll
        for (int r = 0; r < REP; ++r)
#pragma unroll
            for (int k = 0; k < S::EPL / 2; ++k) {
                O2[r][k].x += __shfl_xor_sync(0xffffffffu, O2[r][k].x, m);
                O2[r][k].y += __shfl_xor_sync(0xffffffffu, O2[r][k].y, m);
            }
    // row sums and V-bias sums over the lanes of each row
#pragma unroll
    for (int m = REP; m < 32; m <<= 1) Ssum += __shfl_xor_sync(0xffffffffu, Ssum, m);
    float *sOB = sQS;   // [row][group] totals (the q-group sums are no longer needed)
    __syncwarp();
    for (int g = 0; g < NG; ++g) {
        float x = sOBl[g * 32 + lane];
#pragma unroll
        for (int m = REP; m < 32; m <<= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
        if (lane < REP) sOB[lane * NG + g] = x;
    }
    __syncwarp();
    float Mr[REP], Sr[REP];
#pragma unroll
    for (int r = 0; r < REP; ++r) {
        Mr[r] = __shfl_sync(0xffffffffu, M, r);
        Sr[r] = __shfl_sync(0xffffffffu, Ssum, r);
    }
    if (tv == 0 && pv_live) {
        const int dl = wl * S::EPL;   // first output dimension of the lane
#pragma unroll
        for (int r = 0; r < REP; ++r) {
            if (r >= nrow) break;
            const int q = q0 + r;
            const float ob = sOB[r * NG + g_v];
            if (a.nwg == 1) {
                float c = 1.0f, sf = Sr[r];
                if (a.has_sinks) {
                    const float sk = kLog2e * __ldg(a.sinks + (q % a.nQ));
                    const float mf = fmaxf(Mr[r], sk);
                    c = Mr[r] == -INFINITY ? 0.0f : ex2(Mr[r] - mf);
                    sf = Sr[r] * c + ex2(sk - mf);
                }
                const float f = sf > 0.0f ? c / sf : 0.0f;
#pragma unroll
                for (int k = 0; k < S::EPL / 2; ++k) {
                    st_out<T>(a.out, static_cast<size_t>(q) * dim + dl + 2 * k, (O2[r][k].x + ob) * f, a.out_f32);
                    st_out<T>(a.out, static_cast<size_t>(q) * dim + dl + 2 * k + 1, (O2[r][k].y + ob) * f, a.out_f32);
                }
            } else {
                float2 *po = reinterpret_cast<float2 *>(a.part_o + (static_cast<size_t>(split) * a.rows + q) * dim + dl);
#pragma unroll
                for (int k = 0; k < S::EPL / 2; ++k) po[k] = make_float2(O2[r][k].x + ob, O2[r][k].y + ob);
            }
        }
    }
    if (a.nwg > 1 && lane < nrow)
        reinterpret_cast<float2 *>(a.part_ml)[static_cast<size_t>(split) * a.rows + q0 + lane] = make_float2(Ssum, M);
}

template <int BITS, typename T, int DIMC, int GC>
cudaError_t launch_one(const QuantArgs &a, cudaStream_t s) {
    auto kern = quant_kernel<BITS, T, DIMC, GC>;
    const size_t smem = quant_layout(a.wpt, a.ng, Shape<BITS, DIMC>::CH).total;
    static unsigned long long done = 0;
    cudaError_t e = set_smem_limit_once(kern, kQuantMaxSmem, &done);
    if (e != cudaSuccess) return e;
    kern<<<dim3(a.nwg * a.n_rg, a.kv_rows), 32, smem, s>>>(a);
    count_launch();
    return cudaGetLastError();
}

template <int BITS, typename T, int DIMC, int GC>
int occupancy_one(size_t smem) {
    auto kern = quant_kernel<BITS, T, DIMC, GC>;
    static unsigned long long done = 0;
    if (set_smem_limit_once(kern, kQuantMaxSmem, &done) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 32, smem) != cudaSuccess) return 0;
    return n;
}

// Exact-shape instances exist for group size 64 at every capacity.
inline bool quant_exact(int dim, int G) { return G == 64 && dim == quant_dim_capacity(dim); }

template <int BITS, typename T, int DIMC>
cudaError_t launch_dimc(const QuantArgs &a, cudaStream_t s) {
    if (quant_exact(a.dim, a.G)) return launch_one<BITS, T, DIMC, 64>(a, s);
    return launch_one<BITS, T, DIMC, 0>(a, s);
}

template <int BITS, typename T>
cudaError_t launch_t(const QuantArgs &a, cudaStream_t s) {
    const int dimc = quant_dim_capacity(a.dim);
    if (dimc == 64) return launch_dimc<BITS, T, 64>(a, s);
    if (dimc == 128) return launch_dimc<BITS, T, 128>(a, s);
    if (dimc == 256) return launch_dimc<BITS, T, 256>(a, s);
    return launch_dimc<BITS, T, 512>(a, s);
}

template <int BITS>
cudaError_t launch_bits(const QuantArgs &a, cudaStream_t s) {
    return a.t_is_bf16 ? launch_t<BITS, __nv_bfloat16>(a, s) : launch_t<BITS, __half>(a, s);
}

template <int BITS, typename T, int DIMC>
int occupancy_dimc(bool exact, size_t smem) {
    return exact ? occupancy_one<BITS, T, DIMC, 64>(smem) : occupancy_one<BITS, T, DIMC, 0>(smem);
}

template <int BITS, typename T>
int occupancy_t(int dimc, bool exact, size_t smem) {
    if (dimc == 64) return occupancy_dimc<BITS, T, 64>(exact, smem);
    if (dimc == 128) return occupancy_dimc<BITS, T, 128>(exact, smem);
    if (dimc == 256) return occupancy_dimc<BITS, T, 256>(exact, smem);
    return occupancy_dimc<BITS, T, 512>(exact, smem);
}

template <int BITS>
int occupancy_bits(int dim, int ng) {
    const int dimc = quant_dim_capacity(dim);
    const bool exact = quant_exact(dim, dim / ng);
    const size_t smem = quant_layout(dim * BITS / 32, ng, quant_chunk_tokens(dim, BITS)).total;
    const int a = occupancy_t<BITS, __half>(dimc, exact, smem), b = occupancy_t<BITS, __nv_bfloat16>(dimc, exact, smem);
    return a < b ? a : b;
}

}  // namespace quant
}  // namespace ta
