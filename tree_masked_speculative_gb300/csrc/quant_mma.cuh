// Attention over an affine-quantized K/V cache with warp-level tensor-core
// MMAs (mma.sync m16n8k16, f16 operands, f32 accumulation): the kernel for
// fewer than 16 query rows per KV row.  Included by quant_mma_b4.cu and
// quant_mma_b8.cu, which instantiate it.
//
// What it computes is the quantized-KV attention of quant_kernel.cuh
// (metaltile-std flash_quantized_sdpa.rs: k = s * code + b per group, q
// multiplied by `scale`, window / bool mask / float mask / sinks), with the
// draft-tree gate of quant_sdpa_fwd_tree.
//
// Why MMAs with 4 query rows: on the CUDA cores every code costs a decode and
// a multiply-add per query row, which for 4 rows keeps the FP32 pipe busier
// than HBM.  Here the multiply-adds go to the tensor core, whose rate dwarfs
// what 4 rows need, and a code costs about one integer instruction to decode.
// The same work split (a CTA per KV row, row group of 4 query rows and token
// split) and chunk staging as quant_kernel.cuh, in two forms: one warp doing
// every phase (up to 32 packed words per token) or a score warp handing P to a
// value warp (wider tokens).  In the MMA fragments lane = quad gq = lane / 4
// and position tq = lane % 4:
//  * scores S = Q K^T per chunk: A = Q (M = 16 rows: query row r of a
//    dimension in scale group g sits in row 4 * (g % 4) + r, so one MMA keeps
//    the partial sums of four groups apart), held as f16 scaled per row by a
//    power of two (exact for f16 and bf16 queries); B = the K codes as exact
//    f16 subnormals (code * 2^-24, one AND per two codes), each lane taking a
//    quarter of its key's packed words; the group scales and the bias term
//    sum_g b_g * sum_{d in g} q_d are applied to the f32 sums;
//  * online softmax (log2 units, lazy running max) on the score fragments;
//  * O^T = V^T P^T: A = V dequantized to f16 (s * code + b, one rounding:
//    byte permutes pair two tokens' codes, a magic-exponent OR makes them
//    f16, one subtract and one fused multiply-add per pair), B = P as two f16
//    terms P_hi + P_lo in the 8 columns (4 rows x 2 terms).  The score
//    accumulator fragments of two 8-key blocks are exactly the B fragment of a
//    16-token block, so P never leaves the registers.
#pragma once

#include "quant_kernel.cuh"

namespace ta {
namespace quant {

// D += A B, m16n8k16, f16 inputs, f32 accumulators (register fragments).
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

template <int BITS, int DIMC>
struct MmaShape {
    static constexpr int WPTC = DIMC * BITS / 32;          // packed words per token
    static constexpr int CH = WPTC <= 32 ? 32 : 16;        // tokens per chunk (as quant_chunk_tokens)
    static constexpr int KB = DIMC / 16;                   // score K-blocks = value M-blocks
    static constexpr int NB = CH / 8;                      // score N-blocks (8 keys) per chunk
    static constexpr int VB = CH / 16;                     // value K-blocks (16 tokens) per chunk
    static constexpr int KW = WPTC / 4;                    // K words per lane per key (a quarter)
    static constexpr int VW = WPTC / 8;                    // V words per lane per token (an eighth)
    static_assert(KW >= 1 && VW >= 1 && CH % 16 == 0, "shape");
};

// A fragment of V^T for value M-block mb (16 dimensions) and one 16-token
// block: w[k][u] are the lane's V words u of the block's tokens T0, T1 (k 0,
// 1) and T2, T3 (k 2, 3); sbA[u] / sbB[u] the f16 {s, s} / {b, b} pairs of
// (T0, T1) / (T2, T3) in word u's scale group.  Each register pairs two
// tokens' codes of one dimension (a byte permute), made f16 by an OR under the
// exponent of 1024 (low nibble or byte) or 64 (high nibble), then s * c + b
// rounded once.  ar: a0a1 (row gq, T0 T1), a2a3 (gq + 8, T0 T1), a4a5 (gq,
// T2 T3), a6a7 (gq + 8, T2 T3); row gq is the lower code of its byte (4-bit)
// or byte 2 (mb % 2) (8-bit), row gq + 8 the next dimension.
template <int BITS, int VW>
__device__ __forceinline__ void qmma_v_frag(const uint32_t (&w)[4][VW], const uint2 (&sbA)[VW],
                                            const uint2 (&sbB)[VW], int mb, uint32_t (&ar)[4]) {
    const __half2 k1024 = __float2half2_rn(1024.0f), k64 = __float2half2_rn(64.0f);
    if constexpr (BITS == 4) {
        const int u = mb >> 2, bi = mb & 3;
        const uint32_t sel = static_cast<uint32_t>(bi | (bi << 4) | ((4 + bi) << 8) | ((4 + bi) << 12));
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {   // tokens (T0, T1), then (T2, T3)
            const uint32_t y = __byte_perm(w[2 * hb][u], w[2 * hb + 1][u], sel);
            const uint2 sb = hb ? sbB[u] : sbA[u];
            const __half2 clo = __hsub2(bits_h2((y & 0x000F000Fu) | 0x64006400u), k1024);
            const __half2 chi = __hsub2(bits_h2((y & 0x00F000F0u) | 0x54005400u), k64);
            ar[2 * hb] = h2_bits(__hfma2(clo, bits_h2(sb.x), bits_h2(sb.y)));       // M row gq
            ar[2 * hb + 1] = h2_bits(__hfma2(chi, bits_h2(sb.x), bits_h2(sb.y)));   // M row gq + 8
        }
    } else {
        const int u = mb >> 1, b0 = 2 * (mb & 1);
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            const uint2 sb = hb ? sbB[u] : sbA[u];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {   // byte b0 -> M row gq, b0 + 1 -> gq + 8
                const int bi = b0 + hr;
                const uint32_t sel = static_cast<uint32_t>(bi | (bi << 4) | ((4 + bi) << 8) | ((4 + bi) << 12));
                const uint32_t y = __byte_perm(w[2 * hb][u], w[2 * hb + 1][u], sel);
                const __half2 cc = __hsub2(bits_h2((y & 0x00FF00FFu) | 0x64006400u), k1024);
                ar[2 * hb + hr] = h2_bits(__hfma2(cc, bits_h2(sb.x), bits_h2(sb.y)));
            }
        }
    }
}

// Shared-memory layout: the two staging groups of quant_layout, then the
// kernel's own arrays.
struct QmmaLayout {
    QuantLayout st;
    int qa, qs, qf, ksf, kbias, vsb, pslot, ml, bars, total;
};
// Hand-off slot from the score warp to the value warp: the B fragments of P
// ([16-token block][register][lane]), the per-row rescale factors of O, and
// whether the chunk has any live (row, token) pair.
struct QmmaPSlot {
    uint32_t pf[2][2][32];
    float alpha[4];
    int live;
};
// two_warp: room for the score-to-value hand-off (the two-warp form only).
__host__ __device__ inline QmmaLayout qmma_layout(int wpt, int ng, int ch, int dimc, int nacc, int ns,
                                                  bool two_warp) {
    QmmaLayout M;
    M.st = quant_layout(wpt, ng, ch, ns);
    int o = M.st.v0 + ns * M.st.v_stage;
    M.qa = quant_take(&o, nacc * (dimc / 16) * 32 * 16);   // Q A-fragments [acc][kblock][lane] uint4
    M.qs = quant_take(&o, 4 * ng * 4 + 16);                // [row][group] scale*log2e * sum q, then 2^e per row
    M.qf = quant_take(&o, 4 * dimc * 2);                   // q rows scaled by 2^e, f16 (setup)
    M.ksf = quant_take(&o, ch * ng * 4);                   // [token][group] K scale, f32
    M.kbias = quant_take(&o, ch * 4 * 4);                  // [token][row] score bias term
    M.vsb = quant_take(&o, ng * (ch / 2) * 8);             // [group][token pair] {s, s}, {b, b} f16
    M.pslot = quant_take(&o, two_warp ? 2 * static_cast<int>(sizeof(QmmaPSlot)) : 0);
    M.ml = quant_take(&o, two_warp ? 9 * 4 : 0);           // [row] M, [row] S, abort flag
    M.bars = quant_take(&o, (ns + (two_warp ? 4 : 0)) * 8);   // stages (, P full x 2, P empty x 2)
    M.total = o;
    return M;
}

// Staged chunks in flight (each chunk's K, scale / bias runs, masks and V).
constexpr int kQmmaStages = 2;
// Kernel form of a shape: one warp per CTA up to 32 packed words per token
// (quant_mma1_kernel), else two (quant_mma_kernel); each measured faster there
// (at 32 words the one-warp form took 34.8 against 39.2 us on an 8-bit dim-128
// workload, 54.7 against 55.8 on a 4-bit dim-256 one, and 26.9 against 26.2
// with both masks; at 64 words the two-warp form wins).
template <int WPTC>
struct QmmaForm {
    static constexpr bool one_warp = WPTC <= 32;
    static constexpr int threads = one_warp ? 32 : 64;
};

// Accumulator sets of the score MMA: four scale groups per set.
__host__ __device__ inline int qmma_nacc(int ng) { return (ng + 3) / 4; }

// The phases of a warp-MMA chunk, shared by the one-warp and the two-warp
// forms (each a warp's view: lane = quad gq, position tq).  MASKED: the call
// passes a bool or a float mask (instances without one carry no mask code).
template <int BITS, typename T, int DIMC, int GC, bool MASKED>
struct QmmaPhases {
    using S = MmaShape<BITS, DIMC>;
    static constexpr int CH = S::CH, KB = S::KB, NB = S::NB, VB = S::VB, KW = S::KW, VW = S::VW;
    static constexpr int NG = DIMC / GC;
    static constexpr int NACC = (NG + 3) / 4;
    static constexpr int WPT = S::WPTC;
    static constexpr int QPL = DIMC / 32;   // query elements per lane per row

    const QuantArgs &a;
    const QuantLayout &L;
    uint4 *sQA;
    float *sQS;
    __half *sQF;
    float *sKsf, *sKbias;
    uint2 *sVSB;
    int lane, gq, tq, q0, nrow, N;

    __device__ __forceinline__ int r_l() const { return gq & 3; }   // query row of the score fragments

    // The 4 query rows, element lane + 32 k per lane (issued before anything waits).
    __device__ __forceinline__ void load_q(uint16_t (&qraw)[REP][QPL]) const {
        const uint16_t *qg = reinterpret_cast<const uint16_t *>(a.queries);
#pragma unroll
        for (int r = 0; r < REP; ++r)
#pragma unroll
            for (int k = 0; k < QPL; ++k)
                qraw[r][k] = r < nrow ? __ldg(qg + static_cast<size_t>(q0 + r) * DIMC + lane + 32 * k)
                                      : static_cast<uint16_t>(0);
    }

    // Ancestor bitset of the lane's row's node for a parent-array draft tree (0 without one).
    __device__ __forceinline__ uint32_t tree_bits() const {
        if (a.tree_ql <= 0) return 0u;
        const uint32_t mine = quant_tree_ancestors(lane < a.tree_ql ? __ldg(a.tree_parents + lane) : -1, a.tree_ql);
        return __shfl_sync(0xffffffffu, mine, (q0 + r_l()) % a.tree_ql);
    }

    // Per-row power-of-two scale 2^e (max |q| 2^e in [2^14, 2^15)), group sums
    // (scale * log2(e) * sum_{d in g} q_d), the scaled rows in shared memory and
    // from them the lane's score A-fragments: a0a1 (row gq, slots 0, 1), a2a3
    // (gq + 8, 0, 1), a4a5 (gq, 2, 3), a6a7 (gq + 8, 2, 3) of accumulator set
    // acc and K-block v.  Returns the score scale of the lane's row,
    // scale * log2(e) * 2^24 (subnormal codes) / 2^e.
    __device__ __forceinline__ float setup_scores(const uint16_t (&qraw)[REP][QPL]) const {
        const float qscale = a.scale * kLog2e;
        float *sE2 = sQS + REP * NG;   // 2^e per row
#pragma unroll
        for (int r = 0; r < REP; ++r) {
            float qv[QPL];
            float mx = 0.0f;
#pragma unroll
            for (int k = 0; k < QPL; ++k) {
                qv[k] = t2f<T>(qraw[r][k]);
                mx = fmaxf(mx, fabsf(qv[k]));
            }
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
            int e = 0;
            if (mx > 0.0f) e = 14 - (static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu) - 127);
            const float e2 = ldexpf(1.0f, max(-100, min(100, e)));
            if (lane == 0) sE2[r] = e2;
#pragma unroll
            for (int k = 0; k < QPL; ++k) sQF[r * DIMC + lane + 32 * k] = __float2half_rn(qv[k] * e2);
#pragma unroll
            for (int g = 0; g < NG; ++g) {   // element k is in group 32 k / GC
                float x = 0.0f;
#pragma unroll
                for (int k = 0; k < QPL; ++k)
                    if ((32 * k) / GC == g) x += qv[k];
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
                if (lane == 0) sQS[r * NG + g] = qscale * x;
            }
        }
        __syncwarp();
        // The lane's k-slots of K-block v (k = 2 tq, 2 tq + 1, 2 tq + 8,
        // 2 tq + 9) are four consecutive dimensions d0 .. d0 + 3 of one scale
        // group, the codes the K decode puts there (4-bit: nibbles 4 (v % 2) ..
        // of word tq KW + v / 2; 8-bit: word tq KW + v): slots 0, 1 = d0,
        // d0 + 2 and slots 2, 3 = d0 + 1, d0 + 3 (for 4-bit codes the high
        // nibbles, decoded as 16 * code, so q / 16 there).  One 8-byte load per
        // M row.  Setup code runs once per CTA: the acc loop stays rolled
        // (little code to fetch cold).
        constexpr float fhi = BITS == 4 ? 1.0f / 16.0f : 1.0f;
#pragma unroll 1
        for (int acc = 0; acc < NACC; ++acc)
#pragma unroll 4
            for (int v = 0; v < KB; ++v) {
                const int d0 = BITS == 4 ? 8 * (tq * KW + v / 2) + 4 * (v % 2) : 4 * (tq * KW + v);
                const int g = d0 / GC;
                uint32_t reg[4];
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {   // M row gq, then gq + 8
                    const int m = gq + 8 * hr;
                    uint2 x = make_uint2(0u, 0u);
                    if (g / 4 == acc && (m >> 2) == g % 4)
                        x = *reinterpret_cast<const uint2 *>(sQF + (m & 3) * DIMC + d0);
                    reg[hr] = __byte_perm(x.x, x.y, 0x5410u);   // (d0, d0 + 2)
                    if constexpr (BITS == 4) {
                        const float2 lo = __half22float2(bits_h2(x.x)), hi = __half22float2(bits_h2(x.y));
                        reg[2 + hr] = h2_bits(__floats2half2_rn(lo.y * fhi, hi.y * fhi));   // (d0 + 1, d0 + 3) / 16
                    } else {
                        reg[2 + hr] = __byte_perm(x.x, x.y, 0x7632u);   // (d0 + 1, d0 + 3)
                    }
                }
                sQA[(acc * KB + v) * 32 + lane] = make_uint4(reg[0], reg[1], reg[2], reg[3]);
            }
        __syncwarp();
        return qscale * 16777216.0f / sE2[r_l()];
    }

    // Group sums of the row of this lane's score-bias entries (row = lane % 4).
    __device__ __forceinline__ void bias_sums(float (&qs_l)[NG]) const {
#pragma unroll
        for (int g = 0; g < NG; ++g) qs_l[g] = sQS[(lane & 3) * NG + g];
    }

    // Gates of the lane's (row r_l, key) score slots, key 8 nb + 2 tq + e of the
    // chunk at token t0; returns whether any slot of the warp is live.
    __device__ __forceinline__ bool gates(const unsigned char *st, int t0, uint32_t tree_bits,
                                          bool (&live)[NB][2]) const {
        const uint32_t *sMb = reinterpret_cast<const uint32_t *>(st + L.mb);
        const int tree_lo = N - a.tree_ql;
        bool any = false;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int tk = 8 * nb + 2 * tq + e;
                const int t = t0 + tk;
                bool g = r_l() < nrow && t >= a.t_lo && t < N;
                if (MASKED && g && a.mbool != nullptr) g = sMb[r_l() * CH + tk] != 0u;
                if (g && a.tree_ql > 0 && t >= tree_lo) g = (tree_bits >> (t - tree_lo)) & 1u;
                live[nb][e] = g;
                any |= g;
            }
        return __any_sync(0xffffffffu, any);
    }

    // Per-chunk tables, each lane filling fixed entries: K scales in f32 [t][g],
    // the score bias per (token, row) [t][r] (row = lane % 4), and the V scale /
    // bias pairs of token pairs (2p, 2p + 1) in f16 [g][p].  Each is loaded
    // (k_load, v_load) before any is stored (k_store, v_store), so the loads
    // of a warp doing both are all in flight at once.
    static constexpr int NKS = (CH * NG + 31) / 32, NKB = CH * REP / 32, NVP = (NG * (CH / 2) + 31) / 32;
    struct KRaw {
        uint16_t ks[NKS], kb[NKB][NG];
    };
    struct VRaw {
        uint16_t vs[NVP][2], vb[NVP][2];
    };
    __device__ __forceinline__ void k_load(const unsigned char *st, KRaw &r) const {
        const uint16_t *sKs = reinterpret_cast<const uint16_t *>(st + L.ks);
        const uint16_t *sKb = reinterpret_cast<const uint16_t *>(st + L.kb);
#pragma unroll
        for (int j = 0; j < NKS; ++j) {
            const int idx = lane + 32 * j;
            r.ks[j] = idx < CH * NG ? sKs[idx] : static_cast<uint16_t>(0);
        }
#pragma unroll
        for (int j = 0; j < NKB; ++j) {
            const int t = (lane + 32 * j) / REP;
#pragma unroll
            for (int g = 0; g < NG; ++g) r.kb[j][g] = sKb[t * NG + g];
        }
    }
    __device__ __forceinline__ void k_store(const KRaw &r, const float (&qs_l)[NG]) const {
#pragma unroll
        for (int j = 0; j < NKS; ++j)
            if (lane + 32 * j < CH * NG) sKsf[lane + 32 * j] = t2f<T>(r.ks[j]);
#pragma unroll
        for (int j = 0; j < NKB; ++j) {
            float x = 0.0f;
#pragma unroll
            for (int g = 0; g < NG; ++g) x = fmaf(t2f<T>(r.kb[j][g]), qs_l[g], x);
            sKbias[lane + 32 * j] = x;
        }
    }
    __device__ __forceinline__ void v_load(const unsigned char *st, VRaw &r) const {
        const uint16_t *sVs = reinterpret_cast<const uint16_t *>(st + L.vs);
        const uint16_t *sVb = reinterpret_cast<const uint16_t *>(st + L.vb);
#pragma unroll
        for (int j = 0; j < NVP; ++j) {
            const int idx = lane + 32 * j;
            const int g = idx / (CH / 2), p = idx % (CH / 2);
            const bool in = idx < NG * (CH / 2);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                r.vs[j][e] = in ? sVs[(2 * p + e) * NG + g] : static_cast<uint16_t>(0);
                r.vb[j][e] = in ? sVb[(2 * p + e) * NG + g] : static_cast<uint16_t>(0);
            }
        }
    }
    __device__ __forceinline__ void v_store(const VRaw &r) const {
#pragma unroll
        for (int j = 0; j < NVP; ++j)
            if (lane + 32 * j < NG * (CH / 2)) {
                const __half2 sp = __floats2half2_rn(t2f<T>(r.vs[j][0]), t2f<T>(r.vs[j][1]));
                const __half2 bp = __floats2half2_rn(t2f<T>(r.vb[j][0]), t2f<T>(r.vb[j][1]));
                sVSB[lane + 32 * j] = make_uint2(h2_bits(sp), h2_bits(bp));
            }
    }

    // Scores of the chunk in stage st: the lane's quarter of key 8 nb + gq, all
    // K-blocks, S = Q K^T per accumulator set; then the scale groups apart and
    // the two halves of the quad pair (lanes gq and gq ^ 4 hold the other
    // groups of the same row); live slots get scale * sum + bias (+ float mask)
    // in log2 units.
    __device__ __forceinline__ void scores(const unsigned char *st, float alpha_l, const bool (&live)[NB][2],
                                           float (&lg)[NB][2]) const {
        const uint32_t *sK = reinterpret_cast<const uint32_t *>(st + L.k);
        const uint16_t *sMf = reinterpret_cast<const uint16_t *>(st + L.mf);
        uint32_t kw[NB][KW];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const uint32_t *src = sK + (8 * nb + gq) * WPT + tq * KW;
            if constexpr (KW % 4 == 0) {
#pragma unroll
                for (int u = 0; u < KW; u += 4) {
                    const uint4 x = *reinterpret_cast<const uint4 *>(src + u);
                    kw[nb][u] = x.x; kw[nb][u + 1] = x.y; kw[nb][u + 2] = x.z; kw[nb][u + 3] = x.w;
                }
            } else if constexpr (KW == 2) {
                const uint2 x = *reinterpret_cast<const uint2 *>(src);
                kw[nb][0] = x.x; kw[nb][1] = x.y;
            } else {
#pragma unroll
                for (int u = 0; u < KW; ++u) kw[nb][u] = src[u];
            }
        }
        float sacc[NB][NACC][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int acc = 0; acc < NACC; ++acc)
#pragma unroll
                for (int e = 0; e < 4; ++e) sacc[nb][acc][e] = 0.0f;
#pragma unroll
        for (int v = 0; v < KB; ++v) {
            uint4 af[NACC];
#pragma unroll
            for (int acc = 0; acc < NACC; ++acc) af[acc] = sQA[(acc * KB + v) * 32 + lane];
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                uint32_t b0, b1;
                if constexpr (BITS == 4) {
                    // bytes (2, 3) or (0, 1) of the word into the two halves
                    const uint32_t w = kw[nb][v / 2];
                    const uint32_t y = __byte_perm(w, 0u, (v & 1) ? 0x3322u : 0x1100u);
                    b0 = y & 0x000F000Fu;   // nibbles 0, 2 of the pair: code * 2^-24
                    b1 = y & 0x00F000F0u;   // nibbles 1, 3: 16 * code * 2^-24
                } else {
                    const uint32_t w = kw[nb][v];
                    b0 = w & 0x00FF00FFu;               // bytes 0, 2
                    b1 = __byte_perm(w, 0u, 0x4341u);   // bytes 1, 3
                }
#pragma unroll
                for (int acc = 0; acc < NACC; ++acc)
                    mma16816(sacc[nb][acc], af[acc].x, af[acc].y, af[acc].z, af[acc].w, b0, b1);
            }
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int tk = 8 * nb + 2 * tq + e;
                float x = 0.0f;
#pragma unroll
                for (int acc = 0; acc < NACC; ++acc) {
                    const int glo = 4 * acc + (gq >> 2), ghi = 4 * acc + 2 + (gq >> 2);   // c0/c1, c2/c3 rows
                    if (glo < NG) x = fmaf(sKsf[tk * NG + glo], sacc[nb][acc][e], x);
                    if (NG > 2 && ghi < NG) x = fmaf(sKsf[tk * NG + ghi], sacc[nb][acc][2 + e], x);
                }
                x += __shfl_xor_sync(0xffffffffu, x, 16);
                if (live[nb][e]) {
                    float v = fmaf(alpha_l, x, sKbias[tk * REP + r_l()]);
                    if (MASKED && a.mfloat != nullptr) v = fmaf(kLog2e, t2f<T>(sMf[r_l() * CH + tk]), v);
                    lg[nb][e] = v;
                }
            }
    }

    // Online softmax of row r_l (log2 units), lazy running max: M only moves
    // when a score exceeds it by more than kSlack.  Returns whether any row's
    // max moved (warp-uniform); alpha is then the factor the lane's row's O
    // (and S, rescaled here) is multiplied by, else 1.
    __device__ __forceinline__ bool update_max(const float (&lg)[NB][2], float &Mrow, float &Ssum,
                                               float &alpha) const {
        alpha = 1.0f;
        bool grow = false;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) grow |= lg[nb][0] > Mrow + kSlack || lg[nb][1] > Mrow + kSlack;
        if (!__any_sync(0xffffffffu, grow)) return false;
        float cmax = -INFINITY;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) cmax = fmaxf(cmax, fmaxf(lg[nb][0], lg[nb][1]));
        cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 1));
        cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 2));
        const float m_new = fmaxf(Mrow, cmax);
        alpha = m_new == Mrow ? 1.0f : ex2(Mrow - m_new);   // 0 while M = -inf
        Mrow = m_new;
        Ssum *= alpha;
        return true;
    }

    // B fragments of P (lanes gq < 4 P_hi, gq >= 4 P_lo) and the row sums.
    __device__ __forceinline__ void p_frags(const float (&lg)[NB][2], float Mrow, float &Ssum,
                                            uint32_t (&pf)[VB][2]) const {
        const bool lo_term = gq >= 4;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            float p[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                p[e] = Mrow == -INFINITY ? 0.0f : ex2(lg[nb][e] - Mrow);
                Ssum += p[e];
            }
            const __half2 hi = __floats2half2_rn(p[0], p[1]);
            uint32_t f = h2_bits(hi);
            if (lo_term) {
                const float2 hf = __half22float2(hi);
                f = h2_bits(__floats2half2_rn(p[0] - hf.x, p[1] - hf.y));
            }
            pf[nb >> 1][nb & 1] = f;
        }
    }

    // O^T columns of this lane: n = 2 tq, 2 tq + 1 -> rows (2 tq) % 4, (2 tq) % 4 + 1.
    __device__ __forceinline__ static void rescale_o(float (&O)[KB][4], float al0, float al1) {
#pragma unroll
        for (int mb = 0; mb < KB; ++mb) {
            O[mb][0] *= al0;
            O[mb][1] *= al1;
            O[mb][2] *= al0;
            O[mb][3] *= al1;
        }
    }

    // O^T += V^T P^T per 16-token block of the chunk whose V words are at sV
    // (the V table of the chunk stored).
    __device__ __forceinline__ void pv(const uint32_t *sV, const uint32_t (&pf)[VB][2], float (&O)[KB][4]) const {
        int vgrp[VW];   // scale groups of the lane's V words gq * VW .. + VW
#pragma unroll
        for (int u = 0; u < VW; ++u) vgrp[u] = ((gq * VW + u) * (32 / BITS)) / GC;
#pragma unroll
        for (int kb = 0; kb < VB; ++kb) {
            // tokens of the fragment: (T0, T1) = 16 kb + 2 tq + {0, 1}, (T2, T3) = + 8
            const int tA = 16 * kb + 2 * tq, tB = tA + 8;
            uint32_t w[4][VW];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int t = (k < 2 ? tA : tB) + (k & 1);
                const uint32_t *src = sV + t * WPT + gq * VW;
                if constexpr (VW % 4 == 0) {
#pragma unroll
                    for (int u = 0; u < VW; u += 4) {
                        const uint4 x = *reinterpret_cast<const uint4 *>(src + u);
                        w[k][u] = x.x; w[k][u + 1] = x.y; w[k][u + 2] = x.z; w[k][u + 3] = x.w;
                    }
                } else if constexpr (VW == 2) {
                    const uint2 x = *reinterpret_cast<const uint2 *>(src);
                    w[k][0] = x.x; w[k][1] = x.y;
                } else {
                    w[k][0] = src[0];
                }
            }
            uint2 sbA[VW], sbB[VW];
#pragma unroll
            for (int u = 0; u < VW; ++u) {
                sbA[u] = sVSB[vgrp[u] * (CH / 2) + tA / 2];
                sbB[u] = sVSB[vgrp[u] * (CH / 2) + tB / 2];
            }
#pragma unroll
            for (int mb = 0; mb < KB; ++mb) {
                uint32_t ar[4];
                qmma_v_frag<BITS, VW>(w, sbA, sbB, mb, ar);
                // A regs: a0a1 (row gq, T0 T1), a2a3 (gq + 8, T0 T1), a4a5 (gq, T2 T3), a6a7 (gq + 8, T2 T3)
                mma16816(O[mb], ar[0], ar[1], ar[2], ar[3], pf[kb][0], pf[kb][1]);
            }
        }
    }

    // Output of the rows: O^T columns P_hi + P_lo (tq, tq + 2) added; lanes tq 0
    // and 1 hold rows 2 tq, 2 tq + 1 (c0 / c2 row 2 tq, c1 / c3 row 2 tq + 1).
    // Mr / Sr: the rows' final running max and sum.  One split: out = O / S
    // with the sink; else the split's partial O.
    __device__ __forceinline__ void write_out(float (&O)[KB][4], const float (&Mr)[2], const float (&Sr)[2],
                                              int split) const {
#pragma unroll
        for (int mb = 0; mb < KB; ++mb)
#pragma unroll
            for (int e = 0; e < 4; ++e) O[mb][e] += __shfl_xor_sync(0xffffffffu, O[mb][e], 2);
        if (tq >= 2) return;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int r = 2 * tq + k;
            if (r >= nrow) continue;
            const int q = q0 + r;
            float f = 1.0f;
            if (a.nwg == 1) {
                float cs = 1.0f, sf = Sr[k];
                if (a.has_sinks) {
                    const float sk = kLog2e * __ldg(a.sinks + (q % a.nQ));
                    const float mf = fmaxf(Mr[k], sk);
                    cs = Mr[k] == -INFINITY ? 0.0f : ex2(Mr[k] - mf);
                    sf = Sr[k] * cs + ex2(sk - mf);
                }
                f = sf > 0.0f ? cs / sf : 0.0f;
            }
#pragma unroll
            for (int mb = 0; mb < KB; ++mb) {
                // M row gq of block mb: the low code of its byte, M row gq + 8 the next dimension
                int d;
                if constexpr (BITS == 4) d = 8 * (gq * VW + (mb >> 2)) + 2 * (mb & 3);
                else d = 4 * (gq * VW + (mb >> 1)) + 2 * (mb & 1);
                const float x0 = O[mb][k], x1 = O[mb][2 + k];
                if (a.nwg == 1) {
                    st_out<T>(a.out, static_cast<size_t>(q) * DIMC + d, x0 * f, a.out_f32);
                    st_out<T>(a.out, static_cast<size_t>(q) * DIMC + d + 1, x1 * f, a.out_f32);
                } else {
                    *reinterpret_cast<float2 *>(a.part_o + (static_cast<size_t>(split) * a.rows + q) * DIMC + d) =
                        make_float2(x0, x1);
                }
            }
        }
    }

    // Copies of a chunk's runs.  A full chunk whose runs are 16-byte aligned:
    // one bulk copy per run, each issued by a lane of its own in the same
    // instruction - lane 0 the K words (when this warp copies them), lanes 1-4
    // the K / V scale and bias runs, then one lane per bool-mask and float-mask
    // row - after lane 0 has posted the byte count; the lanes' cp.async
    // arrivals then complete at once (measured against the lanes' 16-byte
    // cp.async of the runs: 28.4 against 28.3 us on the 4-bit dim-128 workload,
    // 34.0 against 34.7 on an 8-bit dim-128 one, 52.6 against 54.6 on a 4-bit
    // dim-256 one).  Other chunks take the staging of quant_kernel.cuh.
    struct CopyPlan {
        const unsigned char *src;   // this lane's run at token 0 (nullptr: none)
        uint32_t stride, bytes, dst, tx;
        bool bulk, with_k;
    };
    __device__ __forceinline__ CopyPlan copy_plan(int kv, bool with_k) const {
        CopyPlan cp{nullptr, 0u, 0u, 0u, 0u, false, with_k};
        {
            cp.bulk = a.al_sb && (a.mbool == nullptr || a.al_mb) && (a.mfloat == nullptr || a.al_mf);
            const size_t kv0 = static_cast<size_t>(kv) * N;
            const int nb_rows = a.mbool != nullptr ? nrow : 0, nf_rows = a.mfloat != nullptr ? nrow : 0;
            if (lane == 0) {
                if (with_k) {
                    cp.src = reinterpret_cast<const unsigned char *>(a.kp + kv0 * WPT);
                    cp.stride = WPT * 4;
                    cp.dst = L.k;
                }
            } else if (lane <= 4) {
                const void *base = lane == 1 ? a.ks : lane == 2 ? a.kb : lane == 3 ? a.vs : a.vb;
                cp.src = reinterpret_cast<const unsigned char *>(static_cast<const uint16_t *>(base) + kv0 * NG);
                cp.stride = NG * 2;
                cp.dst = lane == 1 ? L.ks : lane == 2 ? L.kb : lane == 3 ? L.vs : L.vb;
            } else if (lane < 5 + nb_rows) {   // bool-mask rows 0 .. nrow - 1
                const int r = lane - 5;
                cp.src = reinterpret_cast<const unsigned char *>(a.mbool + static_cast<size_t>(q0 + r) * N);
                cp.stride = 4;
                cp.dst = L.mb + r * CH * 4;
            } else if (lane < 5 + nb_rows + nf_rows) {   // float-mask rows
                const int r = lane - 5 - nb_rows;
                cp.src = reinterpret_cast<const unsigned char *>(static_cast<const uint16_t *>(a.mfloat) +
                                                                 static_cast<size_t>(q0 + r) * N);
                cp.stride = 2;
                cp.dst = L.mf + r * CH * 2;
            }
            cp.bytes = cp.stride * CH;
            cp.tx = CH * ((with_k ? WPT * 4 : 0) + 4 * NG * 2 + nb_rows * 4 + nf_rows * 2);
        }
        return cp;
    }
    // Group A of chunk c into stage b (the K tile only when the plan has it).
    __device__ __forceinline__ void issue_runs(const CopyPlan &cp, const QuantStager<CH> &stg, unsigned char *smem,
                                               uint64_t *bars, int c, int b) const {
        const int t0 = c * CH;
        if (cp.bulk && t0 + CH <= N) {
            unsigned char *st = smem + L.a0 + b * L.a_stage;
            if (lane == 0) {
                if (cp.with_k) mbar_arrive_expect_tx(&bars[b], cp.tx);
                else mbar_expect_tx(&bars[b], cp.tx);
            }
            __syncwarp();
            if (cp.src != nullptr)
                bulk_load(st + cp.dst, cp.src + static_cast<size_t>(t0) * cp.stride, cp.bytes, &bars[b]);
            cp_arrive_noinc(&bars[b]);
        } else {
            stg.issue_a(c, b);
        }
    }
    // The V tile of chunk c into stage b: its bytes posted (no arrival) before
    // group A's arrivals, so the phase cannot complete without them.
    __device__ __forceinline__ void issue_v(unsigned char *smem, uint64_t *bars, int kv, int c, int b) const {
        if (lane == 0) {
            const int t0 = c * CH;
            const uint32_t vbytes = static_cast<uint32_t>(min(CH, N - t0) * WPT * 4);
            mbar_expect_tx(&bars[b], vbytes);
            bulk_load(smem + L.v0 + b * L.v_stage, a.vp + (static_cast<size_t>(kv) * N + t0) * WPT, vbytes, &bars[b]);
        }
    }
    // The K tile of chunk c into stage b (the expect-tx arrive is one of the
    // stage barrier's 33): the two-warp form's score warp.
    __device__ __forceinline__ void issue_k(unsigned char *smem, uint64_t *bars, int kv, int c, int b) const {
        if (lane == 0) {
            const int t0 = c * CH;
            const uint32_t kbytes = static_cast<uint32_t>(min(CH, N - t0) * WPT * 4);
            mbar_arrive_expect_tx(&bars[b], kbytes);
            bulk_load(smem + L.a0 + b * L.a_stage + L.k, a.kp + (static_cast<size_t>(kv) * N + t0) * WPT, kbytes,
                      &bars[b]);
        }
    }
};

// One-warp form (shapes of up to 32 packed words per token, where it measured
// faster than the two-warp form): one warp per CTA does every phase of a chunk
// in turn and issues every copy itself.
template <int BITS, typename T, int DIMC, int GC, bool MASKED>
__global__ void __launch_bounds__(32, 12) quant_mma1_kernel(const QuantArgs a) {
    using P = QmmaPhases<BITS, T, DIMC, GC, MASKED>;
    constexpr int CH = P::CH, NB = P::NB, VB = P::VB, KB = P::KB, NG = P::NG, NS = kQmmaStages;
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x, tq = lane & 3;
    const int rg = blockIdx.x % a.n_rg, split = blockIdx.x / a.n_rg, kv = blockIdx.y;
    const int q0 = kv * a.rep + rg * REP;
    const int nrow = min(REP, a.rep - rg * REP);
    const QmmaLayout M = qmma_layout(P::WPT, NG, CH, DIMC, P::NACC, NS, false);
    const QuantLayout &L = M.st;
    const P ph{a, L, reinterpret_cast<uint4 *>(smem + M.qa), reinterpret_cast<float *>(smem + M.qs),
               reinterpret_cast<__half *>(smem + M.qf), reinterpret_cast<float *>(smem + M.ksf),
               reinterpret_cast<float *>(smem + M.kbias), reinterpret_cast<uint2 *>(smem + M.vsb),
               lane, lane >> 2, tq, q0, nrow, a.N};
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + M.bars);
    const int c_begin = a.c_lo + static_cast<int>((static_cast<long long>(split) * a.nch) / a.nwg);
    const int c_end = a.c_lo + static_cast<int>((static_cast<long long>(split + 1) * a.nch) / a.nwg);
    const int nc = c_end - c_begin;

    uint16_t qraw[REP][P::QPL];
    ph.load_q(qraw);
    const uint32_t tree_bits = ph.tree_bits();
    if (lane == 0) {
        // stage k: lane 0's expect-tx arrive + one cp.async arrive per lane; the
        // V tile's bytes are posted on the same barrier
        for (int k = 0; k < NS; ++k) mbar_init(&bars[k], 33);
        fence_mbar_init();
    }
    __syncwarp();
    const QuantStager<CH> stg{a, L, smem, bars, P::WPT, NG, kv, q0, nrow, lane, NS, true};
    const typename P::CopyPlan cp = ph.copy_plan(kv, true);
    auto issue = [&](int c, int b) {
        ph.issue_v(smem, bars, kv, c, b);
        ph.issue_runs(cp, stg, smem, bars, c, b);
    };
    int issued = 0, done = 0;
    for (; issued < NS && issued < nc; ++issued) issue(c_begin + issued, issued % NS);
    const float alpha_l = ph.setup_scores(qraw);
    float qs_l[NG];
    ph.bias_sums(qs_l);

    float Mrow = -INFINITY, Ssum = 0.0f;   // online softmax of row r_l (log2 units)
    float O[KB][4];
#pragma unroll
    for (int mb = 0; mb < KB; ++mb)
#pragma unroll
        for (int e = 0; e < 4; ++e) O[mb][e] = 0.0f;

    bool ok = true;
    for (int i = 0; i < nc; ++i) {
        const int c = c_begin + i, b = i % NS;
        if (!wait_warp(&bars[b], static_cast<uint32_t>(i / NS) & 1u, i == 0 ? a.first_wait_polls : kQuantWaitPolls)) {
            ok = false;
            break;
        }
        ++done;
        __syncwarp();
        const unsigned char *st = smem + L.a0 + b * L.a_stage;
        bool live[NB][2];
        const bool chunk_live = ph.gates(st, c * CH, tree_bits, live);
        float lg[NB][2];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) lg[nb][0] = lg[nb][1] = -INFINITY;
        if (chunk_live) {
            typename P::KRaw kr;
            typename P::VRaw vr;
            ph.k_load(st, kr);
            ph.v_load(st, vr);
            ph.k_store(kr, qs_l);
            ph.v_store(vr);
            __syncwarp();
            ph.scores(st, alpha_l, live, lg);
        }
        float alpha;
        if (ph.update_max(lg, Mrow, Ssum, alpha)) {   // a row's running max moved
            const int r0 = (2 * tq) & 3;
            P::rescale_o(O, __shfl_sync(0xffffffffu, alpha, 4 * r0), __shfl_sync(0xffffffffu, alpha, 4 * (r0 + 1)));
        }
        if (chunk_live) {
            uint32_t pf[VB][2];
            ph.p_frags(lg, Mrow, Ssum, pf);
            ph.pv(reinterpret_cast<const uint32_t *>(smem + L.v0 + b * L.v_stage), pf, O);
        }
        __syncwarp();
        if (issued < nc) { issue(c_begin + issued, issued % NS); ++issued; }   // stage b is free
    }
    pdl_launch_dependents();   // the merge may start launching; it waits for this grid to finish
    if (!ok) {
        // a copy never completed: report it, let the issued copies land (bounded) and leave
        if (lane == 0 && a.err != nullptr) atomicOr(a.err, 1);
        for (; done < issued; ++done) wait_warp(&bars[done % NS], static_cast<uint32_t>(done / NS) & 1u);
        return;
    }
    // row sums over the quad's keys; the rows' statistics from lanes 4 r
    Ssum += __shfl_xor_sync(0xffffffffu, Ssum, 1);
    Ssum += __shfl_xor_sync(0xffffffffu, Ssum, 2);
    float Mr[2], Sr[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int r = (2 * tq + k) & 3;
        Mr[k] = __shfl_sync(0xffffffffu, Mrow, 4 * r);
        Sr[k] = __shfl_sync(0xffffffffu, Ssum, 4 * r);
    }
    const float s_row = __shfl_sync(0xffffffffu, Ssum, 4 * (lane & 3));
    const float m_row = __shfl_sync(0xffffffffu, Mrow, 4 * (lane & 3));
    ph.write_out(O, Mr, Sr, split);
    if (a.nwg > 1 && lane < nrow)
        reinterpret_cast<float2 *>(a.part_ml)[static_cast<size_t>(split) * a.rows + q0 + lane] =
            make_float2(s_row, m_row);
}

// Two-warp form (wider tokens), one (KV row, row group, token split) per CTA:
//  * warp 0 (scores): gates, the K tables, S = Q K^T, the online softmax and
//    the B fragments of P, handed to warp 1 through a double-buffered slot in
//    shared memory (P, the per-row rescale factors of O, the chunk's
//    liveness); it issues the chunks' K tiles;
//  * warp 1 (values): issues the copies of a chunk's scale / bias runs, masks
//    and V tile (all on the stage's barrier, NS chunks ahead), rescales O,
//    builds the V table, accumulates O^T += V^T P^T and writes the output.
// The two work on different chunks at the same time.
template <int BITS, typename T, int DIMC, int GC, bool MASKED>
__global__ void __launch_bounds__(64, 8) quant_mma_kernel(const QuantArgs a) {
    using P = QmmaPhases<BITS, T, DIMC, GC, MASKED>;
    constexpr int CH = P::CH, NB = P::NB, VB = P::VB, KB = P::KB, NG = P::NG, NS = kQmmaStages;
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = static_cast<int>(threadIdx.x) >> 5, lane = static_cast<int>(threadIdx.x) & 31;
    const int tq = lane & 3;
    const int rg = blockIdx.x % a.n_rg, split = blockIdx.x / a.n_rg, kv = blockIdx.y;
    const int q0 = kv * a.rep + rg * REP;
    const int nrow = min(REP, a.rep - rg * REP);
    const QmmaLayout M = qmma_layout(P::WPT, NG, CH, DIMC, P::NACC, NS, true);
    const QuantLayout &L = M.st;
    const P ph{a, L, reinterpret_cast<uint4 *>(smem + M.qa), reinterpret_cast<float *>(smem + M.qs),
               reinterpret_cast<__half *>(smem + M.qf), reinterpret_cast<float *>(smem + M.ksf),
               reinterpret_cast<float *>(smem + M.kbias), reinterpret_cast<uint2 *>(smem + M.vsb),
               lane, lane >> 2, tq, q0, nrow, a.N};
    QmmaPSlot *sPS = reinterpret_cast<QmmaPSlot *>(smem + M.pslot);
    float *sML = reinterpret_cast<float *>(smem + M.ml);   // [row] M, then [row] S
    volatile int *sAbort = reinterpret_cast<volatile int *>(smem + M.ml + 8 * 4);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + M.bars);
    uint64_t *p_full = bars + NS, *p_empty = bars + NS + 2;
    const int c_begin = a.c_lo + static_cast<int>((static_cast<long long>(split) * a.nch) / a.nwg);
    const int c_end = a.c_lo + static_cast<int>((static_cast<long long>(split + 1) * a.nch) / a.nwg);
    const int nc = c_end - c_begin;

    if (threadIdx.x == 0) {
        // stage k: warp 0's expect-tx arrive for the K tile + one cp.async
        // arrive per lane of warp 1 (scale runs, masks; the V tile's bytes are
        // posted on the same barrier before them)
        for (int k = 0; k < NS; ++k) mbar_init(&bars[k], 33);
        for (int k = 0; k < 2; ++k) {
            mbar_init(&p_full[k], 1);
            mbar_init(&p_empty[k], 1);
        }
        *sAbort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    bool ok = true;
    float O[KB][4];   // warp 1: O^T fragments (M rows = dimensions, columns = rows x {P_hi, P_lo})
#pragma unroll
    for (int mb = 0; mb < KB; ++mb)
#pragma unroll
        for (int e = 0; e < 4; ++e) O[mb][e] = 0.0f;

    if (warp == 1) {
        // ================================================================ values
        const QuantStager<CH> stg{a, L, smem, bars, P::WPT, NG, kv, q0, nrow, lane, NS, false};
        const typename P::CopyPlan cp = ph.copy_plan(kv, false);
        auto issue = [&](int c, int b) {
            ph.issue_v(smem, bars, kv, c, b);
            ph.issue_runs(cp, stg, smem, bars, c, b);
        };
        int issued = 0, done = 0;
        for (; issued < NS && issued < nc; ++issued) issue(c_begin + issued, issued % NS);
        const int r0 = (2 * tq) & 3;   // rows of this lane's O^T columns: r0, r0 + 1
        for (int i = 0; i < nc && ok; ++i) {
            const int b = i % NS, slot = i & 1;
            if (!wait_warp(&bars[b], static_cast<uint32_t>(i / NS) & 1u,
                           i == 0 ? a.first_wait_polls : kQuantWaitPolls) ||
                !wait_warp(&p_full[slot], static_cast<uint32_t>(i >> 1) & 1u)) {
                ok = false;
                break;
            }
            ++done;
            const QmmaPSlot &ps = sPS[slot];
            const float al0 = ps.alpha[r0], al1 = ps.alpha[r0 + 1];
            if (__any_sync(0xffffffffu, al0 != 1.0f || al1 != 1.0f)) P::rescale_o(O, al0, al1);
            if (ps.live) {
                typename P::VRaw vr;
                ph.v_load(smem + L.a0 + b * L.a_stage, vr);
                ph.v_store(vr);
                __syncwarp();
                uint32_t pf[VB][2];
#pragma unroll
                for (int kb = 0; kb < VB; ++kb) {
                    pf[kb][0] = ps.pf[kb][0][lane];
                    pf[kb][1] = ps.pf[kb][1][lane];
                }
                ph.pv(reinterpret_cast<const uint32_t *>(smem + L.v0 + b * L.v_stage), pf, O);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_empty[slot]);   // the slot and the stage's reads are done
            if (issued < nc) { issue(c_begin + issued, issued % NS); ++issued; }   // stage b is free
        }
        if (!ok) {
            // a wait gave up: report it, let the issued copies land (bounded) and leave
            if (lane == 0) {
                *sAbort = 1;
                if (a.err != nullptr) atomicOr(a.err, 1);
            }
            for (; done < issued; ++done) wait_warp(&bars[done % NS], static_cast<uint32_t>(done / NS) & 1u);
        }
    } else {
        // ================================================================ scores
        uint16_t qraw[REP][P::QPL];
        ph.load_q(qraw);
        // the K tiles, NS chunks ahead, each once this warp is done with the stage's K tile
        int k_issued = 0;
        for (; k_issued < NS && k_issued < nc; ++k_issued) ph.issue_k(smem, bars, kv, c_begin + k_issued, k_issued % NS);
        const uint32_t tree_bits = ph.tree_bits();
        const float alpha_l = ph.setup_scores(qraw);
        float qs_l[NG];
        ph.bias_sums(qs_l);

        float Mrow = -INFINITY, Ssum = 0.0f;   // online softmax of row r_l (log2 units)
        for (int i = 0; i < nc && ok; ++i) {
            const int c = c_begin + i, b = i % NS, slot = i & 1;
            if (!wait_warp(&bars[b], static_cast<uint32_t>(i / NS) & 1u,
                           i == 0 ? a.first_wait_polls : kQuantWaitPolls)) {
                ok = false;
                break;
            }
            const unsigned char *st = smem + L.a0 + b * L.a_stage;
            bool live[NB][2];
            const bool chunk_live = ph.gates(st, c * CH, tree_bits, live);
            float lg[NB][2];
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) lg[nb][0] = lg[nb][1] = -INFINITY;
            if (chunk_live) {
                typename P::KRaw kr;
                ph.k_load(st, kr);
                ph.k_store(kr, qs_l);
                __syncwarp();
                ph.scores(st, alpha_l, live, lg);
            }
            __syncwarp();
            if (k_issued < nc) {   // this chunk's K tile is read
                ph.issue_k(smem, bars, kv, c_begin + k_issued, k_issued % NS);
                ++k_issued;
            }
            float alpha;
            ph.update_max(lg, Mrow, Ssum, alpha);
            uint32_t pf[VB][2];
#pragma unroll
            for (int kb = 0; kb < VB; ++kb) pf[kb][0] = pf[kb][1] = 0u;
            if (chunk_live) ph.p_frags(lg, Mrow, Ssum, pf);
            // hand P, the rescale factors and the liveness to warp 1
            if (!wait_warp(&p_empty[slot], (static_cast<uint32_t>(i >> 1) & 1u) ^ 1u)) {
                ok = false;
                break;
            }
            QmmaPSlot &ps = sPS[slot];
#pragma unroll
            for (int kb = 0; kb < VB; ++kb) {
                ps.pf[kb][0][lane] = pf[kb][0];
                ps.pf[kb][1][lane] = pf[kb][1];
            }
            if (tq == 0 && (lane >> 2) < 4) ps.alpha[lane >> 2] = alpha;
            if (lane == 0) ps.live = chunk_live ? 1 : 0;
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[slot]);
        }
        if (!ok && lane == 0) {
            *sAbort = 1;
            if (a.err != nullptr) atomicOr(a.err, 1);
        }
        // row statistics for the epilogue: S summed over the quad's keys
        Ssum += __shfl_xor_sync(0xffffffffu, Ssum, 1);
        Ssum += __shfl_xor_sync(0xffffffffu, Ssum, 2);
        if (tq == 0 && (lane >> 2) < 4) {
            sML[lane >> 2] = Mrow;
            sML[4 + (lane >> 2)] = Ssum;
        }
    }
    pdl_launch_dependents();   // the merge may start launching; it waits for this grid to finish
    __syncthreads();
    if (*sAbort != 0) return;
    if (warp == 0) {
        if (a.nwg > 1 && lane < nrow)
            reinterpret_cast<float2 *>(a.part_ml)[static_cast<size_t>(split) * a.rows + q0 + lane] =
                make_float2(sML[4 + lane], sML[lane]);
        return;
    }
    float Mr[2], Sr[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int r = (2 * tq + k) & 3;
        Mr[k] = sML[r];
        Sr[k] = sML[4 + r];
    }
    ph.write_out(O, Mr, Sr, split);
}

template <int BITS, int DIMC, int GC>
inline size_t mma_smem_bytes() {
    using S = MmaShape<BITS, DIMC>;
    return static_cast<size_t>(qmma_layout(S::WPTC, DIMC / GC, S::CH, DIMC, qmma_nacc(DIMC / GC), kQmmaStages,
                                           !QmmaForm<S::WPTC>::one_warp).total);
}

template <int BITS, typename T, int DIMC, int GC, bool MASKED>
constexpr auto mma_kernel_of() {
    if constexpr (QmmaForm<MmaShape<BITS, DIMC>::WPTC>::one_warp) return quant_mma1_kernel<BITS, T, DIMC, GC, MASKED>;
    else return quant_mma_kernel<BITS, T, DIMC, GC, MASKED>;
}

template <int BITS, typename T, int DIMC, int GC, bool MASKED>
cudaError_t mma_launch_masked(const QuantArgs &a, cudaStream_t s) {
    auto kern = mma_kernel_of<BITS, T, DIMC, GC, MASKED>();
    constexpr int threads = QmmaForm<MmaShape<BITS, DIMC>::WPTC>::threads;
    static unsigned long long done = 0;
    cudaError_t e = set_smem_limit_once(kern, kQuantMaxSmem, &done);
    if (e != cudaSuccess) return e;
    kern<<<dim3(a.nwg * a.n_rg, a.kv_rows), threads, mma_smem_bytes<BITS, DIMC, GC>(), s>>>(a);
    count_launch();
    return cudaGetLastError();
}

template <int BITS, typename T, int DIMC, int GC>
cudaError_t mma_launch_one(const QuantArgs &a, cudaStream_t s) {
    if (a.mbool != nullptr || a.mfloat != nullptr) return mma_launch_masked<BITS, T, DIMC, GC, true>(a, s);
    return mma_launch_masked<BITS, T, DIMC, GC, false>(a, s);
}

template <int BITS, typename T, int DIMC, int GC, bool MASKED>
int mma_occupancy_masked() {
    auto kern = mma_kernel_of<BITS, T, DIMC, GC, MASKED>();
    constexpr int threads = QmmaForm<MmaShape<BITS, DIMC>::WPTC>::threads;
    static unsigned long long done = 0;
    if (set_smem_limit_once(kern, kQuantMaxSmem, &done) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, mma_smem_bytes<BITS, DIMC, GC>()) !=
        cudaSuccess)
        return 0;
    return n;
}

// Resident CTAs per SM: the smaller of the two instances (the split count
// does not depend on which masks a call passes).
template <int BITS, typename T, int DIMC, int GC>
int mma_occupancy_one() {
    const int u = mma_occupancy_masked<BITS, T, DIMC, GC, false>(), m = mma_occupancy_masked<BITS, T, DIMC, GC, true>();
    return u < m ? u : m;
}

// Instances: head dimension 64, 128 or 256 exactly, group size 32 or 64
// (quant_mma_shape_ok); anything else is not launched.
template <int BITS, typename T>
cudaError_t mma_launch_t(const QuantArgs &a, cudaStream_t s) {
    const bool g32 = a.G == 32;
    if (a.dim == 64) return g32 ? mma_launch_one<BITS, T, 64, 32>(a, s) : mma_launch_one<BITS, T, 64, 64>(a, s);
    if (a.dim == 128) return g32 ? mma_launch_one<BITS, T, 128, 32>(a, s) : mma_launch_one<BITS, T, 128, 64>(a, s);
    return g32 ? mma_launch_one<BITS, T, 256, 32>(a, s) : mma_launch_one<BITS, T, 256, 64>(a, s);
}

template <int BITS>
cudaError_t mma_launch_bits(const QuantArgs &a, cudaStream_t s) {
    return a.t_is_bf16 ? mma_launch_t<BITS, __nv_bfloat16>(a, s) : mma_launch_t<BITS, __half>(a, s);
}

template <int BITS, typename T>
int mma_occupancy_t(int dim, int G) {
    const bool g32 = G == 32;
    if (dim == 64) return g32 ? mma_occupancy_one<BITS, T, 64, 32>() : mma_occupancy_one<BITS, T, 64, 64>();
    if (dim == 128) return g32 ? mma_occupancy_one<BITS, T, 128, 32>() : mma_occupancy_one<BITS, T, 128, 64>();
    return g32 ? mma_occupancy_one<BITS, T, 256, 32>() : mma_occupancy_one<BITS, T, 256, 64>();
}

template <int BITS>
int mma_occupancy_bits(int dim, int ng) {
    const int G = dim / ng;
    const int a = mma_occupancy_t<BITS, __half>(dim, G), b = mma_occupancy_t<BITS, __nv_bfloat16>(dim, G);
    return a < b ? a : b;
}

}  // namespace quant
}  // namespace ta
