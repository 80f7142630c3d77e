// Quantized-KV main pass on the warp-level tensor-core MMA, 16 query rows per
// warp (the wide form of the warp-MMA kernel, for 16 or more query rows per KV
// row: GQA groups of that size, or the rows of a draft tree being verified).
//
// MLX-style affine codes (w = s * code + b per group of G dimensions, as in
// metaltile-std flash_quantized_sdpa.rs) make each K or V element an integer
// code and its group's (s, b).  The 4-row form (quant_mma.cuh) keeps four
// scale groups apart in the 16 M rows of one score MMA; with 16 rows per warp
// every M row is a query row, so here each score MMA's 16 dimensions lie in
// one scale group instead and the group scale multiplies that group's sums:
//  * scores S = Q K^T per chunk of 32 keys, 8 keys per MMA: A = Q (rows scaled
//    by 2^e_r into f16), B = the K codes as exact f16 subnormals; the lane's
//    k-slots of K-block v are word 4 u + tq of the key's 16-byte run u (u = v
//    / 2 for 4-bit codes, v for 8-bit), fetched with one ldmatrix per key block
//    and scale group; after a group's K-blocks its sums take s_{t,g};
//  * the bias term sum_g b_{t,g} sum_{d in g} q_d and the float mask go into
//    the logits (log2 units); bool mask, window and draft-tree gates;
//  * online softmax of the lane's two rows (gq, gq + 8), lazy running max;
//  * values O^T = V^T P^T: A = V dequantized to f16 (qmma_v_frag, as the 4-row
//    form), B = P^T for 8 rows (rows 0-7 or 8-15), as P_hi + P_lo in two MMAs
//    into the same accumulators; the score accumulators of two 8-key blocks
//    are the B fragments of a 16-token block, so P never leaves registers.
// Staging as the 4-row form: each chunk's K words, scale / bias runs, mask
// rows and V tile on one mbarrier, two chunks ahead.
#pragma once

#include "quant_mma.cuh"

namespace ta {
namespace quant {

constexpr int kQ16Rows = 16;   // query rows of a CTA

template <int BITS, int DIMC>
struct Mma16Shape {
    static constexpr int WPTC = DIMC * BITS / 32;   // packed words per token (8, 16 or 32)
    static constexpr int CH = 32;                   // tokens per chunk
    static constexpr int KB = DIMC / 16;            // score K-blocks = value M-blocks
    static constexpr int NB = CH / 8;               // score N-blocks (8 keys)
    static constexpr int VB = CH / 16;              // value K-blocks (16 tokens)
    static constexpr int KPR = BITS == 4 ? 2 : 1;   // K-blocks per 16-byte run of a key
    static constexpr int VW = WPTC / 8;             // V words per lane per token
    static_assert(WPTC >= 8 && WPTC <= 32 && VW >= 1, "shape");
};

// Shared-memory layout: the staging groups of quant_layout (mask rows for 16
// query rows), then the kernel's own arrays.
struct Q16Layout {
    QuantLayout st;
    int qa, qs, qf, ksf, kbf, vsb, bars, total;
};
__host__ __device__ inline Q16Layout q16_layout(int wpt, int ng, int ch, int dimc, int ns) {
    Q16Layout M;
    M.st = quant_layout(wpt, ng, ch, ns, kQ16Rows);
    int o = M.st.v0 + ns * M.st.v_stage;
    M.qa = quant_take(&o, (dimc / 16) * 32 * 16);          // Q A-fragments [kblock][lane] uint4
    M.qs = quant_take(&o, kQ16Rows * ng * 4 + kQ16Rows * 4);   // [row][group] scale*log2e*sum q, then 2^e per row
    M.qf = quant_take(&o, kQ16Rows * dimc * 2);             // query rows (raw, then scaled f16; setup)
    M.ksf = quant_take(&o, ng * ch * 4);                    // [group][token] K scale, f32
    M.kbf = quant_take(&o, ng * ch * 4);                    // [group][token] K bias, f32
    M.vsb = quant_take(&o, ng * (ch / 2) * 8);              // [group][token pair] {s, s}, {b, b} f16
    M.bars = quant_take(&o, ns * 8);
    M.total = o;
    return M;
}

// ldmatrix of R 8x8 16-bit matrices (R = 1, 2 or 4): lane i gives the row
// address of row i % 8 of matrix i / 8 and receives, of each matrix j, the
// 32-bit word i % 4 of row i / 4 in r[j].
template <int R>
__device__ __forceinline__ void ldsm(uint32_t (&r)[R], uint32_t addr) {
    if constexpr (R == 4)
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(addr));
    else if constexpr (R == 2)
        asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
    else
        asm volatile("ldmatrix.sync.aligned.m8n8.x1.shared.b16 {%0}, [%1];" : "=r"(r[0]) : "r"(addr));
}

// One warp per CTA: (KV row, row group of 16 query rows, token split).
template <int BITS, typename T, int DIMC, int GC, bool MASKED>
__global__ void __launch_bounds__(32, 8) quant_mma16_kernel(const QuantArgs a) {
    using S = Mma16Shape<BITS, DIMC>;
    constexpr int CH = S::CH, KB = S::KB, NB = S::NB, VB = S::VB, VW = S::VW, WPT = S::WPTC;
    constexpr int NG = DIMC / GC, NS = kQmmaStages;
    constexpr int KPG = GC / 16;            // K-blocks per scale group
    constexpr int RPG = KPG / S::KPR;       // 16-byte runs of a key per scale group (1, 2 or 4)
    static_assert(KPG % S::KPR == 0 && (RPG == 1 || RPG == 2 || RPG == 4), "group size");
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = static_cast<int>(threadIdx.x), gq = lane >> 2, tq = lane & 3;
    const int rg = blockIdx.x % a.n_rg, split = blockIdx.x / a.n_rg, kv = blockIdx.y;
    const int q0 = kv * a.rep + rg * kQ16Rows;
    const int nrow = min(kQ16Rows, a.rep - rg * kQ16Rows);
    const int N = a.N;
    const Q16Layout M = q16_layout(WPT, NG, CH, DIMC, NS);
    const QuantLayout &L = M.st;
    uint4 *sQA = reinterpret_cast<uint4 *>(smem + M.qa);
    float *sQS = reinterpret_cast<float *>(smem + M.qs);
    float *sE2 = sQS + kQ16Rows * NG;
    uint16_t *sQF = reinterpret_cast<uint16_t *>(smem + M.qf);
    float *sKsf = reinterpret_cast<float *>(smem + M.ksf);
    float *sKbf = reinterpret_cast<float *>(smem + M.kbf);
    uint2 *sVSB = reinterpret_cast<uint2 *>(smem + M.vsb);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + M.bars);
    const int c_begin = a.c_lo + static_cast<int>((static_cast<long long>(split) * a.nch) / a.nwg);
    const int c_end = a.c_lo + static_cast<int>((static_cast<long long>(split + 1) * a.nch) / a.nwg);
    const int nc = c_end - c_begin;

    if (lane == 0) {
        // stage k: lane 0's expect-tx arrive + one cp.async arrive per lane; the
        // V tile's bytes are posted on the same barrier
        for (int k = 0; k < NS; ++k) mbar_init(&bars[k], 33);
        fence_mbar_init();
    }
    __syncwarp();

    // ---- copies of chunk c into stage b (as the 4-row form): one bulk copy per
    // run of a full chunk whose runs are 16-byte aligned, one lane per copy,
    // else the lanes' cp.async (quant_kernel.cuh); the V tile by one bulk copy
    const QuantStager<CH> stg{a, L, smem, bars, WPT, NG, kv, q0, nrow, lane, NS, true};
    const int nb_rows = (MASKED && a.mbool != nullptr) ? nrow : 0;
    const int nf_rows = (MASKED && a.mfloat != nullptr) ? nrow : 0;
    const bool bulk = a.al_sb && (nb_rows == 0 || a.al_mb) && (nf_rows == 0 || a.al_mf) && 5 + nb_rows + nf_rows <= 32;
    const unsigned char *cp_src = nullptr;
    uint32_t cp_stride = 0u, cp_dst = 0u;
    {
        const size_t kv0 = static_cast<size_t>(kv) * N;
        if (lane == 0) {
            cp_src = reinterpret_cast<const unsigned char *>(a.kp + kv0 * WPT);
            cp_stride = WPT * 4;
            cp_dst = L.k;
        } else if (lane <= 4) {
            const void *base = lane == 1 ? a.ks : lane == 2 ? a.kb : lane == 3 ? a.vs : a.vb;
            cp_src = reinterpret_cast<const unsigned char *>(static_cast<const uint16_t *>(base) + kv0 * NG);
            cp_stride = NG * 2;
            cp_dst = lane == 1 ? L.ks : lane == 2 ? L.kb : lane == 3 ? L.vs : L.vb;
        } else if (MASKED && lane < 5 + nb_rows) {
            const int r = lane - 5;
            cp_src = reinterpret_cast<const unsigned char *>(a.mbool + static_cast<size_t>(q0 + r) * N);
            cp_stride = 4;
            cp_dst = L.mb + r * CH * 4;
        } else if (MASKED && lane < 5 + nb_rows + nf_rows) {
            const int r = lane - 5 - nb_rows;
            cp_src = reinterpret_cast<const unsigned char *>(static_cast<const uint16_t *>(a.mfloat) +
                                                             static_cast<size_t>(q0 + r) * N);
            cp_stride = 2;
            cp_dst = L.mf + r * CH * 2;
        }
    }
    const uint32_t cp_tx = CH * (WPT * 4 + 4 * NG * 2 + nb_rows * 4 + nf_rows * 2);
    auto issue = [&](int c, int b) {
        const int t0 = c * CH;
        if (lane == 0) {
            const uint32_t vbytes = static_cast<uint32_t>(min(CH, N - t0) * WPT * 4);
            mbar_expect_tx(&bars[b], vbytes);
            bulk_load(smem + L.v0 + b * L.v_stage, a.vp + (static_cast<size_t>(kv) * N + t0) * WPT, vbytes, &bars[b]);
        }
        if (bulk && t0 + CH <= N) {
            unsigned char *st = smem + L.a0 + b * L.a_stage;
            if (lane == 0) mbar_arrive_expect_tx(&bars[b], cp_tx);
            __syncwarp();
            if (cp_src != nullptr)
                bulk_load(st + cp_dst, cp_src + static_cast<size_t>(t0) * cp_stride, cp_stride * CH, &bars[b]);
            cp_arrive_noinc(&bars[b]);
        } else {
            stg.issue_a(c, b);
        }
    };
    int issued = 0, done = 0;
    for (; issued < NS && issued < nc; ++issued) issue(c_begin + issued, issued % NS);

    // ---- query rows: lane 2 r + h holds half h of row r; per-row power-of-two
    // scale 2^e (max |q| 2^e in [2^14, 2^15)), group sums scale * log2(e) *
    // sum_{d in g} q_d, the scaled rows in f16, then the score A-fragments
    constexpr int HALF = DIMC / 2;
    const float qscale = a.scale * kLog2e;
    {
        const int r = lane >> 1, h = lane & 1;
        const uint16_t *qg = reinterpret_cast<const uint16_t *>(a.queries) + static_cast<size_t>(q0 + r) * DIMC + h * HALF;
        const bool live = r < nrow;
        // the half-row's elements, two per word (element 2 k in the low half of raw[k])
        uint32_t raw[HALF / 2];
        if (live && (reinterpret_cast<uintptr_t>(a.queries) & 15u) == 0) {
#pragma unroll
            for (int k8 = 0; k8 < HALF / 8; ++k8) {
                const uint4 x = __ldg(reinterpret_cast<const uint4 *>(qg + 8 * k8));
                raw[4 * k8] = x.x; raw[4 * k8 + 1] = x.y; raw[4 * k8 + 2] = x.z; raw[4 * k8 + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int k = 0; k < HALF / 2; ++k)
                raw[k] = live ? static_cast<uint32_t>(__ldg(qg + 2 * k)) | (static_cast<uint32_t>(__ldg(qg + 2 * k + 1)) << 16)
                              : 0u;
        }
        float mx = 0.0f, gs[NG];
#pragma unroll
        for (int g = 0; g < NG; ++g) gs[g] = 0.0f;
#pragma unroll
        for (int k = 0; k < HALF / 2; ++k) {
            const float v0 = t2f<T>(static_cast<uint16_t>(raw[k] & 0xffffu)), v1 = t2f<T>(static_cast<uint16_t>(raw[k] >> 16));
            mx = fmaxf(mx, fmaxf(fabsf(v0), fabsf(v1)));
            const int g = (h * HALF + 2 * k) / GC;   // both elements in one group
#pragma unroll
            for (int gg = 0; gg < NG; ++gg)
                if (gg == g) gs[gg] += v0 + v1;
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
#pragma unroll
        for (int g = 0; g < NG; ++g) gs[g] += __shfl_xor_sync(0xffffffffu, gs[g], 1);
        int e = 0;
        if (mx > 0.0f) e = 14 - (static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu) - 127);
        const float e2 = ldexpf(1.0f, max(-100, min(100, e)));
        if (h == 0) {
            sE2[r] = e2;
#pragma unroll
            for (int g = 0; g < NG; ++g) sQS[r * NG + g] = qscale * gs[g];
        }
        // the half-row scaled by 2^e, in f16, by 16-byte stores
#pragma unroll
        for (int k = 0; k < HALF / 2; ++k) {
            const float v0 = t2f<T>(static_cast<uint16_t>(raw[k] & 0xffffu)), v1 = t2f<T>(static_cast<uint16_t>(raw[k] >> 16));
            raw[k] = h2_bits(__floats2half2_rn(v0 * e2, v1 * e2));
        }
        uint4 *dst = reinterpret_cast<uint4 *>(sQF + r * DIMC + h * HALF);
#pragma unroll
        for (int k8 = 0; k8 < HALF / 8; ++k8)
            dst[k8] = make_uint4(raw[4 * k8], raw[4 * k8 + 1], raw[4 * k8 + 2], raw[4 * k8 + 3]);
    }
    __syncwarp();
    // A-fragments of K-block v: the lane's k-slots (k = 2 tq, 2 tq + 1, 2 tq + 8,
    // 2 tq + 9) are four consecutive dimensions d0 .. d0 + 3 of word 4 u + tq
    // (slots 0, 1 = d0, d0 + 2; slots 2, 3 = d0 + 1, d0 + 3, for 4-bit codes the
    // high nibbles, decoded as 16 * code, so q / 16 there); a0a1 row gq, a2a3
    // row gq + 8 (slots 0, 1), a4a5 / a6a7 the same rows (slots 2, 3)
    {
        constexpr float fhi = BITS == 4 ? 1.0f / 16.0f : 1.0f;
        const __half *qf = reinterpret_cast<const __half *>(sQF);
#pragma unroll 4
        for (int v = 0; v < KB; ++v) {
            const int wd = 4 * (v / S::KPR) + tq;
            const int d0 = BITS == 4 ? 8 * wd + 4 * (v % 2) : 4 * wd;
            uint32_t reg[4];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const uint2 x = *reinterpret_cast<const uint2 *>(qf + (gq + 8 * hr) * DIMC + d0);
                reg[hr] = __byte_perm(x.x, x.y, 0x5410u);   // (d0, d0 + 2)
                if constexpr (BITS == 4) {
                    const float2 lo = __half22float2(bits_h2(x.x)), hi = __half22float2(bits_h2(x.y));
                    reg[2 + hr] = h2_bits(__floats2half2_rn(lo.y * fhi, hi.y * fhi));
                } else {
                    reg[2 + hr] = __byte_perm(x.x, x.y, 0x7632u);   // (d0 + 1, d0 + 3)
                }
            }
            sQA[v * 32 + lane] = make_uint4(reg[0], reg[1], reg[2], reg[3]);
        }
    }
    __syncwarp();
    // the lane's rows gq + 8 h: score scale (scale * log2(e) * 2^24 / 2^e_r),
    // bias-term group sums, draft-tree ancestor bitsets
    float alpha_r[2], qs_r[2][NG];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        alpha_r[h] = qscale * 16777216.0f / sE2[gq + 8 * h];
#pragma unroll
        for (int g = 0; g < NG; ++g) qs_r[h][g] = sQS[(gq + 8 * h) * NG + g];
    }
    uint32_t tbits[2] = {0u, 0u};
    if (a.tree_ql > 0) {
        const uint32_t mine = quant_tree_ancestors(lane < a.tree_ql ? __ldg(a.tree_parents + lane) : -1, a.tree_ql);
#pragma unroll
        for (int h = 0; h < 2; ++h) tbits[h] = __shfl_sync(0xffffffffu, mine, (q0 + gq + 8 * h) % a.tree_ql);
    }
    const int tree_lo = N - a.tree_ql;

    float Mrow[2] = {-INFINITY, -INFINITY}, Ssum[2] = {0.0f, 0.0f};   // rows gq, gq + 8 (log2 units)
    float O[KB][2][4];   // O^T: M-block mb (dimensions) x rows 8 rb .. 8 rb + 7
#pragma unroll
    for (int mb = 0; mb < KB; ++mb)
#pragma unroll
        for (int rb = 0; rb < 2; ++rb)
#pragma unroll
            for (int e = 0; e < 4; ++e) O[mb][rb][e] = 0.0f;

    bool ok = true;
    for (int i = 0; i < nc; ++i) {
        const int c = c_begin + i, b = i % NS, t0 = c * CH;
        if (!wait_warp(&bars[b], static_cast<uint32_t>(i / NS) & 1u, i == 0 ? a.first_wait_polls : kQuantWaitPolls)) {
            ok = false;
            break;
        }
        ++done;
        __syncwarp();
        const unsigned char *st = smem + L.a0 + b * L.a_stage;
        // gates of the lane's slots: [nb][e] = (row gq + 8 (e >> 1), key 8 nb + 2 tq + (e & 1))
        bool live[NB][4];
        bool any = false;
        // a chunk inside the window, before the draft-tree positions and without a
        // bool mask keeps every key of the CTA's rows (the common case)
        const bool plain = !(MASKED && a.mbool != nullptr) && t0 >= a.t_lo && t0 + CH <= N &&
                           (a.tree_ql <= 0 || t0 + CH <= tree_lo);
        if (plain) {
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int e = 0; e < 4; ++e) live[nb][e] = gq + 8 * (e >> 1) < nrow;
            any = true;   // row 0 exists
        } else {
            const uint32_t *sMb = reinterpret_cast<const uint32_t *>(st + L.mb);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = gq + 8 * (e >> 1), tk = 8 * nb + 2 * tq + (e & 1), t = t0 + tk;
                    bool g = r < nrow && t >= a.t_lo && t < N;
                    if (MASKED && g && a.mbool != nullptr) g = sMb[r * CH + tk] != 0u;
                    if (g && a.tree_ql > 0 && t >= tree_lo) g = (tbits[e >> 1] >> (t - tree_lo)) & 1u;
                    live[nb][e] = g;
                    any |= g;
                }
        }
        const bool chunk_live = __any_sync(0xffffffffu, any);
        float lg[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int e = 0; e < 4; ++e) lg[nb][e] = -INFINITY;
        if (chunk_live) {
            // tables: K scales and biases in f32 [group][token], V scale / bias
            // pairs of token pairs in f16 [group][pair]
            {
                const uint16_t *sKs = reinterpret_cast<const uint16_t *>(st + L.ks);
                const uint16_t *sKb = reinterpret_cast<const uint16_t *>(st + L.kb);
                const uint16_t *sVs = reinterpret_cast<const uint16_t *>(st + L.vs);
                const uint16_t *sVb = reinterpret_cast<const uint16_t *>(st + L.vb);
                constexpr int NKT = (CH * NG + 31) / 32, NVP = (NG * (CH / 2) + 31) / 32;
                uint16_t ks[NKT], kb[NKT], vs[NVP][2], vb[NVP][2];
#pragma unroll
                for (int j = 0; j < NKT; ++j) {
                    const int idx = lane + 32 * j, g = idx / CH, t = idx % CH;   // [g][t]
                    ks[j] = idx < CH * NG ? sKs[t * NG + g] : static_cast<uint16_t>(0);
                    kb[j] = idx < CH * NG ? sKb[t * NG + g] : static_cast<uint16_t>(0);
                }
#pragma unroll
                for (int j = 0; j < NVP; ++j) {
                    const int idx = lane + 32 * j, g = idx / (CH / 2), p = idx % (CH / 2);
                    const bool in = idx < NG * (CH / 2);
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        vs[j][e] = in ? sVs[(2 * p + e) * NG + g] : static_cast<uint16_t>(0);
                        vb[j][e] = in ? sVb[(2 * p + e) * NG + g] : static_cast<uint16_t>(0);
                    }
                }
#pragma unroll
                for (int j = 0; j < NKT; ++j)
                    if (lane + 32 * j < CH * NG) {
                        sKsf[lane + 32 * j] = t2f<T>(ks[j]);
                        sKbf[lane + 32 * j] = t2f<T>(kb[j]);
                    }
#pragma unroll
                for (int j = 0; j < NVP; ++j)
                    if (lane + 32 * j < NG * (CH / 2)) {
                        const __half2 sp = __floats2half2_rn(t2f<T>(vs[j][0]), t2f<T>(vs[j][1]));
                        const __half2 bp = __floats2half2_rn(t2f<T>(vb[j][0]), t2f<T>(vb[j][1]));
                        sVSB[lane + 32 * j] = make_uint2(h2_bits(sp), h2_bits(bp));
                    }
            }
            __syncwarp();
            // scores: per scale group, its K-blocks' MMAs, then the group scale
            float x[NB][4];
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int e = 0; e < 4; ++e) x[nb][e] = 0.0f;
            const uint32_t sK = smem_u32(st + L.k);
            const int mrow = lane & 7, mat = min(lane >> 3, RPG - 1);
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                uint32_t kw[NB][RPG];   // word 4 u + tq of key 8 nb + gq, runs u of group g
#pragma unroll
                for (int nb = 0; nb < NB; ++nb)
                    ldsm<RPG>(kw[nb], sK + static_cast<uint32_t>(((8 * nb + mrow) * WPT + 4 * (g * RPG + mat)) * 4));
                float acc[NB][4];
#pragma unroll
                for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[nb][e] = 0.0f;
#pragma unroll
                for (int kl = 0; kl < KPG; ++kl) {
                    const uint4 af = sQA[(g * KPG + kl) * 32 + lane];
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) {
                        uint32_t b0, b1;
                        const uint32_t w = kw[nb][kl / S::KPR];
                        if constexpr (BITS == 4) {
                            const uint32_t y = __byte_perm(w, 0u, (kl & 1) ? 0x3322u : 0x1100u);
                            b0 = y & 0x000F000Fu;   // nibbles 0, 2 of the byte pair: code * 2^-24
                            b1 = y & 0x00F000F0u;   // nibbles 1, 3: 16 * code * 2^-24
                        } else {
                            b0 = w & 0x00FF00FFu;               // bytes 0, 2
                            b1 = __byte_perm(w, 0u, 0x4341u);   // bytes 1, 3
                        }
                        mma16816(acc[nb], af.x, af.y, af.z, af.w, b0, b1);
                    }
                }
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    const float2 s = *reinterpret_cast<const float2 *>(sKsf + g * CH + 8 * nb + 2 * tq);
                    x[nb][0] = fmaf(s.x, acc[nb][0], x[nb][0]);
                    x[nb][1] = fmaf(s.y, acc[nb][1], x[nb][1]);
                    x[nb][2] = fmaf(s.x, acc[nb][2], x[nb][2]);
                    x[nb][3] = fmaf(s.y, acc[nb][3], x[nb][3]);
                }
            }
            // logits of live slots: scale * sum + bias term (+ float mask), log2 units
            const uint16_t *sMf = reinterpret_cast<const uint16_t *>(st + L.mf);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                float bias[2][2];   // [row half][key]
#pragma unroll
                for (int k = 0; k < 2; ++k) bias[0][k] = bias[1][k] = 0.0f;
#pragma unroll
                for (int g = 0; g < NG; ++g) {
                    const float2 kbv = *reinterpret_cast<const float2 *>(sKbf + g * CH + 8 * nb + 2 * tq);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        bias[h][0] = fmaf(kbv.x, qs_r[h][g], bias[h][0]);
                        bias[h][1] = fmaf(kbv.y, qs_r[h][g], bias[h][1]);
                    }
                }
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (live[nb][e]) {
                        const int h = e >> 1, tk = 8 * nb + 2 * tq + (e & 1);
                        float v = fmaf(alpha_r[h], x[nb][e], bias[h][e & 1]);
                        if (MASKED && a.mfloat != nullptr)
                            v = fmaf(kLog2e, t2f<T>(sMf[(gq + 8 * h) * CH + tk]), v);
                        lg[nb][e] = v;
                    }
            }
        }
        // online softmax of the lane's rows (lazy running max, kSlack)
        {
            bool grow = false;
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int e = 0; e < 4; ++e) grow |= lg[nb][e] > Mrow[e >> 1] + kSlack;
            if (__any_sync(0xffffffffu, grow)) {
                float al[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float cmax = -INFINITY;
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) cmax = fmaxf(cmax, fmaxf(lg[nb][2 * h], lg[nb][2 * h + 1]));
                    cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 1));
                    cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 2));
                    const float m_new = fmaxf(Mrow[h], cmax);
                    al[h] = m_new == Mrow[h] ? 1.0f : ex2(Mrow[h] - m_new);   // 0 while M = -inf
                    Mrow[h] = m_new;
                    Ssum[h] *= al[h];
                }
                // O^T columns 2 tq, 2 tq + 1 of row block rb: rows 8 rb + 2 tq + k,
                // whose factor lane 4 (2 tq + k) holds in al[rb]
#pragma unroll
                for (int rb = 0; rb < 2; ++rb) {
                    const float f0 = __shfl_sync(0xffffffffu, al[rb], 8 * tq);
                    const float f1 = __shfl_sync(0xffffffffu, al[rb], 8 * tq + 4);
#pragma unroll
                    for (int mb = 0; mb < KB; ++mb) {
                        O[mb][rb][0] *= f0;
                        O[mb][rb][1] *= f1;
                        O[mb][rb][2] *= f0;
                        O[mb][rb][3] *= f1;
                    }
                }
            }
        }
        if (chunk_live) {
            // B fragments of P^T: [row block][16-token block][P_hi, P_lo][register]
            uint32_t pf[2][VB][2][2];
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float p[2];
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        p[k] = Mrow[h] == -INFINITY ? 0.0f : ex2(lg[nb][2 * h + k] - Mrow[h]);
                        Ssum[h] += p[k];
                    }
                    const __half2 hi = __floats2half2_rn(p[0], p[1]);
                    const float2 hf = __half22float2(hi);
                    pf[h][nb >> 1][0][nb & 1] = h2_bits(hi);
                    pf[h][nb >> 1][1][nb & 1] = h2_bits(__floats2half2_rn(p[0] - hf.x, p[1] - hf.y));
                }
            // O^T += V^T P^T per 16-token block
            const uint32_t *sV = reinterpret_cast<const uint32_t *>(smem + L.v0 + b * L.v_stage);
            int vgrp[VW];   // scale groups of the lane's V words gq * VW .. + VW
#pragma unroll
            for (int u = 0; u < VW; ++u) vgrp[u] = ((gq * VW + u) * (32 / BITS)) / GC;
#pragma unroll
            for (int kb = 0; kb < VB; ++kb) {
                const int tA = 16 * kb + 2 * tq, tB = tA + 8;
                uint32_t w[4][VW];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int t = (k < 2 ? tA : tB) + (k & 1);
                    const uint32_t *src = sV + t * WPT + gq * VW;
                    if constexpr (VW % 4 == 0) {
#pragma unroll
                        for (int u = 0; u < VW; u += 4) {
                            const uint4 xv = *reinterpret_cast<const uint4 *>(src + u);
                            w[k][u] = xv.x; w[k][u + 1] = xv.y; w[k][u + 2] = xv.z; w[k][u + 3] = xv.w;
                        }
                    } else if constexpr (VW == 2) {
                        const uint2 xv = *reinterpret_cast<const uint2 *>(src);
                        w[k][0] = xv.x; w[k][1] = xv.y;
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
#pragma unroll
                    for (int rb = 0; rb < 2; ++rb) {
                        mma16816(O[mb][rb], ar[0], ar[1], ar[2], ar[3], pf[rb][kb][0][0], pf[rb][kb][0][1]);
                        mma16816(O[mb][rb], ar[0], ar[1], ar[2], ar[3], pf[rb][kb][1][0], pf[rb][kb][1][1]);
                    }
                }
            }
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
    // row sums over the quad's keys; the statistics of rows 8 rb + 2 tq + k
    // from lane 4 (2 tq + k)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        Ssum[h] += __shfl_xor_sync(0xffffffffu, Ssum[h], 1);
        Ssum[h] += __shfl_xor_sync(0xffffffffu, Ssum[h], 2);
    }
    if (a.nwg > 1 && tq == 0) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
            if (gq + 8 * h < nrow)
                reinterpret_cast<float2 *>(a.part_ml)[static_cast<size_t>(split) * a.rows + q0 + gq + 8 * h] =
                    make_float2(Ssum[h], Mrow[h]);
    }
#pragma unroll
    for (int rb = 0; rb < 2; ++rb)
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float m = __shfl_sync(0xffffffffu, Mrow[rb], 4 * (2 * tq + k));
            const float sm = __shfl_sync(0xffffffffu, Ssum[rb], 4 * (2 * tq + k));
            const int r = 8 * rb + 2 * tq + k;
            if (r >= nrow) continue;
            const int q = q0 + r;
            float f = 1.0f;
            if (a.nwg == 1) {
                float cs = 1.0f, sf = sm;
                if (a.has_sinks) {
                    const float sk = kLog2e * __ldg(a.sinks + (q % a.nQ));
                    const float mf = fmaxf(m, sk);
                    cs = m == -INFINITY ? 0.0f : ex2(m - mf);
                    sf = sm * cs + ex2(sk - mf);
                }
                f = sf > 0.0f ? cs / sf : 0.0f;
            }
#pragma unroll
            for (int mb = 0; mb < KB; ++mb) {
                // M row gq of block mb: the low code of its byte, M row gq + 8 the next dimension
                int d;
                if constexpr (BITS == 4) d = 8 * (gq * VW + (mb >> 2)) + 2 * (mb & 3);
                else d = 4 * (gq * VW + (mb >> 1)) + 2 * (mb & 1);
                const float x0 = O[mb][rb][k], x1 = O[mb][rb][2 + k];
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

}  // namespace quant
}  // namespace ta

namespace ta {
namespace quant {

template <int BITS, int DIMC, int GC>
inline size_t mma16_smem_bytes() {
    return static_cast<size_t>(
        q16_layout(Mma16Shape<BITS, DIMC>::WPTC, DIMC / GC, Mma16Shape<BITS, DIMC>::CH, DIMC, kQmmaStages).total);
}

template <int BITS, typename T, int DIMC, int GC, bool MASKED>
cudaError_t mma16_launch_masked(const QuantArgs &a, cudaStream_t s) {
    auto kern = quant_mma16_kernel<BITS, T, DIMC, GC, MASKED>;
    static unsigned long long done = 0;
    cudaError_t e = set_smem_limit_once(kern, kQuantMaxSmem, &done);
    if (e != cudaSuccess) return e;
    kern<<<dim3(a.nwg * a.n_rg, a.kv_rows), 32, mma16_smem_bytes<BITS, DIMC, GC>(), s>>>(a);
    count_launch();
    return cudaGetLastError();
}

template <int BITS, typename T, int DIMC, int GC, bool MASKED>
int mma16_occupancy_masked() {
    auto kern = quant_mma16_kernel<BITS, T, DIMC, GC, MASKED>;
    static unsigned long long done = 0;
    if (set_smem_limit_once(kern, kQuantMaxSmem, &done) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 32, mma16_smem_bytes<BITS, DIMC, GC>()) != cudaSuccess)
        return 0;
    return n;
}

template <int BITS, typename T, int DIMC, int GC>
cudaError_t mma16_launch_one(const QuantArgs &a, cudaStream_t s) {
    if (a.mbool != nullptr || a.mfloat != nullptr) return mma16_launch_masked<BITS, T, DIMC, GC, true>(a, s);
    return mma16_launch_masked<BITS, T, DIMC, GC, false>(a, s);
}

template <int BITS, typename T, int DIMC, int GC>
int mma16_occupancy_one() {
    const int u = mma16_occupancy_masked<BITS, T, DIMC, GC, false>();
    const int m = mma16_occupancy_masked<BITS, T, DIMC, GC, true>();
    return u < m ? u : m;
}

// Instances: head dimension 64 or 128, group size 32 or 64 (quant_mma_wide);
// anything else is not launched.
template <int BITS, typename T>
cudaError_t mma16_launch_t(const QuantArgs &a, cudaStream_t s) {
    const bool g32 = a.G == 32;
    if (a.dim == 64) return g32 ? mma16_launch_one<BITS, T, 64, 32>(a, s) : mma16_launch_one<BITS, T, 64, 64>(a, s);
    return g32 ? mma16_launch_one<BITS, T, 128, 32>(a, s) : mma16_launch_one<BITS, T, 128, 64>(a, s);
}

template <int BITS>
cudaError_t mma16_launch_bits(const QuantArgs &a, cudaStream_t s) {
    if ((a.dim != 64 && a.dim != 128) || (a.G != 32 && a.G != 64)) return cudaErrorInvalidValue;
    return a.t_is_bf16 ? mma16_launch_t<BITS, __nv_bfloat16>(a, s) : mma16_launch_t<BITS, __half>(a, s);
}

template <int BITS, typename T>
int mma16_occupancy_t(int dim, int G) {
    const bool g32 = G == 32;
    if (dim == 64) return g32 ? mma16_occupancy_one<BITS, T, 64, 32>() : mma16_occupancy_one<BITS, T, 64, 64>();
    return g32 ? mma16_occupancy_one<BITS, T, 128, 32>() : mma16_occupancy_one<BITS, T, 128, 64>();
}

template <int BITS>
int mma16_occupancy_bits(int dim, int ng) {
    if (ng <= 0 || (dim != 64 && dim != 128)) return 0;
    const int G = dim / ng;
    if (G != 32 && G != 64) return 0;
    const int a = mma16_occupancy_t<BITS, __half>(dim, G), b = mma16_occupancy_t<BITS, __nv_bfloat16>(dim, G);
    return a < b ? a : b;
}

}  // namespace quant
}  // namespace ta
