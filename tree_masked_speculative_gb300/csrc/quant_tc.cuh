// Attention over an affine-quantized K/V cache on the tensor cores (tcgen05).
// Included by quant_tc_b4.cu and quant_tc_b8.cu, which instantiate it.
//
// What it computes is what the CUDA-core kernel computes (metaltile-std
// flash_quantized_sdpa.rs: base, bool-mask and float-mask kernels): element d
// of a K or V token is scale[d / G] * code_d + bias[d / G]; q is scaled by
// `scale` before the dot; window and bool-mask gates; the float mask added to
// the logit; a sink as a virtual key of value 0 (finalisation or merge).
//
// GB300 design.  One CTA = (token split, block of up to RR = 4, 8, 16 or 32
// query rows of one KV row); the token range is walked in 128-token tiles.
//   warp 0      : producer.  Per tile, the packed K words (one bulk copy) into
//                 the K ring; the packed V words, the four scale / bias runs
//                 (bulk copies, or plain loads for a ragged or unaligned tile)
//                 and the rows' bool / float mask runs (per-lane cp.async) into
//                 the V ring.
//   warps 2..9  : decoders, four for K and four for V, each group filling its
//                 own ring of 16 KB chunks ([128 tokens][64 dims], 128-byte
//                 swizzled) in tile order: K as the exact integer codes (byte
//                 permutes under the f16 exponent of 1024, minus 1024), V as
//                 s * code + b rounded once to f16.
//   warp 1      : TMEM owner and score MMA issuer.  Scores transposed, tokens
//                 on the M side: S^T_g = Kcodes_g Q_g'^T per scale group g (M
//                 128 tokens, N = max(16, RR) rows, one f32 accumulator per
//                 group, double buffered).
//   warp 18     : PV MMA issuer: O^T += V^T P^T (M 128 dimensions, N = max(16,
//                 RR) rows, V MN-major, P as two f16 terms from shared memory).
//   warps 10..17: softmax, one thread per (token, half of the rows): logit =
//                 2^e_r * scale * log2(e) * (sum_g s_g S^T_g + b_g * 2^-e_r *
//                 sum_{d in g} q_d) (+ log2(e) * float mask); row maxima by a
//                 warp reduce-scatter and an exchange among the four warps of a
//                 half; lazy running max (moves only by more than 2^8); P in f16
//                 into the A operand of PV; per-lane row sums.  The warp on TMEM
//                 lanes 0..31 of the first half rescales O when a max moves and
//                 writes the rows out.  These warps also stage Q at the start.
// Q is staged once as f16 after scaling each row by a power of two (2^-e_r,
// max |q'| in [2^14, 2^15)), exact for f16 and bf16 queries; K codes enter
// the MMA exactly, so the scores carry only f32 accumulation error; V values
// carry one f16 rounding and P enters as two f16 terms (P_hi + P_lo).  For 4-bit codes the decoded dimensions
// of every 8-dimension word sit in the order 0,4,1,5,2,6,3,7 (one mask-and-or
// per pair); Q follows the same order and O columns are put back on output.
// Every mbarrier wait is bounded; on a timeout the CTA sets bit 0 of the
// error word, drains its copies and MMAs, frees TMEM and exits.
#pragma once

#include <type_traits>

#include "sm100_ptx.cuh"
#include "ta_internal.cuh"

namespace ta {
namespace qtc {

using namespace ta::sm100;

constexpr int kDecWarps = 8;      // decoders: four for K, four for V
constexpr int kDecGroup = 4;
constexpr int kSmWarps = 8;       // softmax: two per TMEM lane quarter, each half of the rows
constexpr int kPvWarp = 2 + kDecWarps + kSmWarps;   // the PV MMA issuer, after the softmax warps
constexpr int kThreads = 32 * (kPvWarp + 1);
constexpr uint32_t kPolls = 1u << 21;     // bound of every wait: tries of up to kSleepNs each
constexpr uint32_t kSleepNs = 1000;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kSlack = 8.0f;      // lazy-max slack (log2 units): P <= 256
constexpr int kMaxRing = kQuantTcMaxRing;

struct Bars {
    uint64_t kfull[kMaxRing], kempty[kMaxRing];
    uint64_t vfull[kMaxRing], vempty[kMaxRing];
    uint64_t dfull[kMaxRing], dempty[kMaxRing];
    uint64_t s_full[2], s_free[2], p_full[2], p_free[2], o_done[2];   // per tile parity
    uint64_t q_ready, drain, drain_pv;
    uint32_t tmem_base;
    volatile int abort_flag;
};
static_assert(sizeof(Bars) <= kQtcBarBytes, "barrier area");

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float t2f(uint16_t bits, bool bf16) {
    return bf16 ? __uint_as_float(static_cast<uint32_t>(bits) << 16) : __half2float(__ushort_as_half(bits));
}
__device__ __forceinline__ __half t2h(uint16_t bits, bool bf16) {
    return bf16 ? __float2half_rn(__uint_as_float(static_cast<uint32_t>(bits) << 16)) : __ushort_as_half(bits);
}
__device__ __forceinline__ void cp16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void note_abort(Bars *b, int *err) {
    b->abort_flag = 1;
    atomicOr(err, 1);
}
// Bounded wait of one thread; false (and the CTA marked aborted) on timeout.
__device__ __forceinline__ bool wait1(Bars *b, uint64_t *bar, uint32_t parity, int *err) {
    if (mbar_try_wait(bar, parity)) return true;      // the common case: the phase is already complete
    if (b->abort_flag) return false;
    if (mbar_wait_sleep(bar, parity, kPolls, kSleepNs)) return true;
    note_abort(b, err);
    return false;
}
// Bounded wait of a whole warp: lane 0 polls (32 polling lanes per warp would
// crowd the shared-memory pipe the working warps use), the warp barrier then
// orders the other lanes after its acquire.  The result is warp-uniform.
__device__ __forceinline__ bool waitw(Bars *b, uint64_t *bar, uint32_t parity, int *err) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = wait1(b, bar, parity, err);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok;
}

// Position of dimension k (0..7) of a 4-bit word in its decoded 8-dimension
// piece (the decode leaves the pairs (c0, c4), (c1, c5), (c2, c6), (c3, c7)).
__device__ __forceinline__ int pos4(int k) { return ((k & 3) << 1) | (k >> 2); }

template <int N>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, uint32_t (&r)[N]);
template <int N>
__device__ __forceinline__ void tmem_stn(uint32_t taddr, const uint32_t (&r)[N]);
template <>
__device__ __forceinline__ void tmem_stn<2>(uint32_t taddr, const uint32_t (&r)[2]) { tmem_st2(taddr, r); }
template <>
__device__ __forceinline__ void tmem_stn<4>(uint32_t taddr, const uint32_t (&r)[4]) { tmem_st4(taddr, r); }
template <>
__device__ __forceinline__ void tmem_stn<8>(uint32_t taddr, const uint32_t (&r)[8]) { tmem_st8(taddr, r); }
template <>
__device__ __forceinline__ void tmem_stn<16>(uint32_t taddr, const uint32_t (&r)[16]) { tmem_st16(taddr, r); }
template <>
__device__ __forceinline__ void tmem_stn<32>(uint32_t taddr, const uint32_t (&r)[32]) { tmem_st32(taddr, r); }
template <>
__device__ __forceinline__ void tmem_ldn<2>(uint32_t taddr, uint32_t (&r)[2]) { tmem_ld2(taddr, r); }
template <>
__device__ __forceinline__ void tmem_ldn<4>(uint32_t taddr, uint32_t (&r)[4]) { tmem_ld4(taddr, r); }
template <>
__device__ __forceinline__ void tmem_ldn<8>(uint32_t taddr, uint32_t (&r)[8]) { tmem_ld8(taddr, r); }
template <>
__device__ __forceinline__ void tmem_ldn<16>(uint32_t taddr, uint32_t (&r)[16]) { tmem_ld16(taddr, r); }
template <>
__device__ __forceinline__ void tmem_ldn<32>(uint32_t taddr, uint32_t (&r)[32]) { tmem_ld32(taddr, r); }

// Reduce-scatter over groups of N lanes (xor 1 .. N/2): lane l returns the
// max (or sum) over its group of value index l % N.  Destroys v.
template <int N, bool MAX>
__device__ __forceinline__ float reduce_scatter(float (&v)[N], int lane) {
#pragma unroll
    for (int s = 0; (1 << s) < N; ++s) {
        const int m = 1 << s;
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int k = 0; k < (N >> s) / 2; ++k) {
            const float send = upper ? v[2 * k] : v[2 * k + 1];
            const float keep = upper ? v[2 * k + 1] : v[2 * k];
            const float got = __shfl_xor_sync(0xffffffffu, send, m);
            v[k] = MAX ? fmaxf(keep, got) : keep + got;
        }
    }
    return v[0];
}

// Decode chunk c (dimensions [64c, 64c + 64)) of a tile's packed words into a
// [128 tokens][64 x f16] 128-byte-swizzled operand chunk: the codes (K) or
// s * code + b (V).  kDecGroup * 32 threads; a 16-byte item is four words of
// a token.
template <int BITS>
__device__ __forceinline__ void decode_chunk(const uint32_t *words, int wpt, int c, unsigned char *dst, int dtid,
                                             bool is_v, const uint16_t *vs, const uint16_t *vb, int ng, int G,
                                             bool bf16) {
    constexpr int DPW = 32 / BITS;          // dimensions per word
    constexpr int IPT = 64 / (4 * DPW);     // items per token and chunk (2 or 4)
    constexpr int PPI = 4 * DPW / 8;        // 16-byte output pieces per item (4 or 2)
    const __half2 k1024 = __float2half2_rn(1024.0f);
    constexpr int NIT = 128 * IPT / (kDecGroup * 32);   // items per thread
#pragma unroll
    for (int i = 0; i < NIT; ++i) {
        const int it = dtid + kDecGroup * 32 * i;
        const int tok = it / IPT, h = it % IPT;
        const uint4 w4 = *reinterpret_cast<const uint4 *>(words + tok * wpt + c * (64 / DPW) + h * 4);
        const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
        __half2 s2 = k1024, b2 = k1024;
        if (is_v) {
            const int g = (c * 64 + h * 4 * DPW) / G;
            s2 = __half2half2(t2h(vs[tok * ng + g], bf16));
            b2 = __half2half2(t2h(vb[tok * ng + g], bf16));
        }
        constexpr int NO = BITS == 4 ? 16 : 8;   // f16 pairs per item
        uint32_t out[NO];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if constexpr (BITS == 4) {
#pragma unroll
                for (int k = 0; k < 4; ++k) out[u * 4 + k] = ((w[u] >> (4 * k)) & 0x000F000Fu) | 0x64006400u;
            } else {
                out[u * 2 + 0] = __byte_perm(w[u], 0x64646464u, 0x5140u);
                out[u * 2 + 1] = __byte_perm(w[u], 0x64646464u, 0x5342u);
            }
        }
#pragma unroll
        for (int e = 0; e < NO; ++e) {
            __half2 x = __hsub2(*reinterpret_cast<__half2 *>(&out[e]), k1024);   // exact code
            if (is_v) x = __hfma2(x, s2, b2);                                   // s * c + b, rounded once
            out[e] = *reinterpret_cast<uint32_t *>(&x);
        }
#pragma unroll
        for (int p = 0; p < PPI; ++p) {
            const int j = h * PPI + p;
            *reinterpret_cast<uint4 *>(dst + tok * 128 + ((j ^ (tok & 7)) << 4)) =
                make_uint4(out[4 * p], out[4 * p + 1], out[4 * p + 2], out[4 * p + 3]);
        }
    }
}

// RR: query rows of a CTA (4, 8, 16 or 32); each softmax lane handles RH =
// RR / 2 of them (two warps per TMEM lane quarter).  The score MMA's N (and
// the Q and score-buffer layout) is RP = max(16, RR), its extra rows zero.
template <int BITS, int RR>
__global__ void __launch_bounds__(kThreads, 1) quant_tc_kernel(const QuantArgs a) {
    constexpr int RP = RR < 16 ? 16 : RR;
    constexpr int RH = RR / 2;
    extern __shared__ __align__(1024) unsigned char smem[];
    // 128-byte-swizzled operands need a 1024-byte-aligned base (the same for
    // every CTA, so a misaligned one stops all of them before any barrier)
    if ((smem_u32(smem) & 1023u) != 0) {
        if (threadIdx.x == 0) atomicOr(a.err, 1);
        return;
    }
    const bool has_mb = a.mbool != nullptr, has_mf = a.mfloat != nullptr;
    const int NG = a.ng, DIM = a.dim, WPT = a.wpt, G = a.G, N = a.N;
    const int ND = a.tc_nd, NK = a.tc_nk, NV = a.tc_nv;
    const QtcLayout L = qtc_layout(RP, DIM, WPT, NG, ND, NK, NV, has_mb, has_mf);
    Bars *bars = reinterpret_cast<Bars *>(smem + L.bars);
    float *sF = reinterpret_cast<float *>(smem + L.rc);      // [RP] 2^e_r * scale * log2(e)
    float *sQG = sF + RP;                                     // [NG][RP] 2^-e_r * sum_{d in g} q_d
    // softmax exchange: row maxima [parity][half][quarter][32], row sums
    // [half][quarter][32], final row maxima [32]
    float *sMax = reinterpret_cast<float *>(smem + L.red);
    float *sSum = sMax + 512;
    float *sMrow = sSum + 256;
    uint32_t *sTree = reinterpret_cast<uint32_t *>(sMrow + 32);   // [32] ancestor bitsets of a draft tree
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, rb = blockIdx.y % a.n_rb, kv = blockIdx.y / a.n_rb;
    const int q0 = kv * a.rep + rb * RR;
    const int rows_here = min(RR, a.rep - rb * RR);
    const int j0 = a.j_lo + static_cast<int>((static_cast<long long>(split) * a.ntile) / a.nwg);
    const int j1 = a.j_lo + static_cast<int>((static_cast<long long>(split + 1) * a.ntile) / a.nwg);
    const int T = j1 - j0;
    const int NCH = DIM / 64;
    const bool bf16 = a.t_is_bf16 != 0;
    int *err = a.err;

    if (warp == 0) {
        // the barriers, initialized by the lanes of warp 0 in parallel
        if (lane < NK) {
            mbar_init(&bars->kfull[lane], 1);
            mbar_init(&bars->kempty[lane], kDecGroup);
        }
        // V slot: the producer's expect-tx arrive, 32 cp.async arrivals, 32 plain arrivals
        if (lane < NV) {
            mbar_init(&bars->vfull[lane], 65);
            mbar_init(&bars->vempty[lane], kDecGroup + kSmWarps);
        }
        if (lane < ND) {
            mbar_init(&bars->dfull[lane], kDecGroup);
            mbar_init(&bars->dempty[lane], 1);
        }
        if (lane < 2) {
            mbar_init(&bars->s_full[lane], 1);
            mbar_init(&bars->s_free[lane], kSmWarps);
            mbar_init(&bars->p_full[lane], kSmWarps);
            mbar_init(&bars->p_free[lane], 1);
            mbar_init(&bars->o_done[lane], 1);
        }
        if (lane == 31) {
            mbar_init(&bars->q_ready, kSmWarps);
            mbar_init(&bars->drain, 1);
            mbar_init(&bars->drain_pv, 1);
            bars->abort_flag = 0;
        }
        fence_mbar_init();
    }
    // the softmax warps fetch their Q rows now, to use them once the barriers exist
    constexpr int RPW = RP / kSmWarps;                  // Q rows staged per softmax warp (2 or 4)
    const int sw = warp - 2 - kDecWarps;                // softmax warp index (0..7 for those warps)
    const int E = DIM / 32;                             // Q elements per lane (2, 4 or 8)
    float qx[RPW][8];
    // the first softmax warp also fetches the draft tree's parent array now
    const int tree_up = (sw == 0 && lane < a.tree_ql) ? __ldg(a.tree_parents + lane) : -1;
    if (sw >= 0 && sw < kSmWarps) {
        const uint16_t *qg = static_cast<const uint16_t *>(a.queries);
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
            const int r = sw + kSmWarps * i;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                qx[i][e] = (e < E && r < rows_here) ? t2f(qg[static_cast<size_t>(q0 + r) * DIM + lane * E + e], bf16)
                                                    : 0.0f;
        }
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, static_cast<uint32_t>(a.tc_cols));
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    // TMEM: O^T (lanes = dimensions of a 128-dimension block, columns = rows),
    // RP columns per block, then the two score buffers
    const int OB = DIM >= 128 ? DIM / 128 : 1;
    const uint32_t tm_o = tmem;
    auto tm_s = [&](int sb) { return tmem + static_cast<uint32_t>(OB * RP + sb * NG * RP); };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int kn = 0, vn = 0;
        const size_t row0 = static_cast<size_t>(kv) * N;
        // scale / bias run k (0..3: K scales, K biases, V scales, V biases): source and slot offset
        auto sb_src = [&](int k) {
            return static_cast<const uint16_t *>(k == 0 ? a.ks : k == 1 ? a.kb : k == 2 ? a.vs : a.vb);
        };
        auto sb_off = [&](int k) { return k == 0 ? L.vks : k == 1 ? L.vkb : k == 2 ? L.vvs : L.vvb; };
        for (int t = 0; t < T; ++t) {
            const int t0 = (j0 + t) * 128;
            const int tval = min(128, N - t0);
            const bool full = tval == 128;
            bool ok = true;
            {
                const int slot = kn % NK;
                if (lane == 0) {
                    ok = wait1(bars, &bars->kempty[slot], (static_cast<uint32_t>(kn / NK) & 1u) ^ 1u, err);
                    if (ok) {
                        const uint32_t bytes = static_cast<uint32_t>(tval * WPT * 4);
                        mbar_arrive_expect_tx(&bars->kfull[slot], bytes);
                        bulk_load(smem + L.k0 + slot * L.kslot, a.kp + (row0 + t0) * WPT, bytes, &bars->kfull[slot]);
                    }
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
                ++kn;
            }
            {
                const int slot = vn % NV;
                unsigned char *st = smem + L.v0 + slot * L.vslot;
                const bool sb_bulk = a.al_sb && full;
                const uint32_t sbb = static_cast<uint32_t>(128 * NG * 2);
                if (lane == 0) {
                    ok = wait1(bars, &bars->vempty[slot], (static_cast<uint32_t>(vn / NV) & 1u) ^ 1u, err);
                    if (ok) {
                        const uint32_t vbytes = static_cast<uint32_t>(tval * WPT * 4);
                        mbar_arrive_expect_tx(&bars->vfull[slot], vbytes + (sb_bulk ? 4 * sbb : 0u));
                        bulk_load(st + L.vw, a.vp + (row0 + t0) * WPT, vbytes, &bars->vfull[slot]);
                        if (sb_bulk)
                            for (int k = 0; k < 4; ++k)
                                bulk_load(st + sb_off(k), sb_src(k) + (row0 + t0) * NG, sbb, &bars->vfull[slot]);
                    }
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
                ++vn;
                if (!sb_bulk) {
                    const int per = 128 * NG, valid = tval * NG;
                    for (int i = lane; i < 4 * per; i += 32) {
                        const int k = i / per, e = i % per;
                        reinterpret_cast<uint16_t *>(st + sb_off(k))[e] =
                            e < valid ? sb_src(k)[(row0 + t0) * NG + e] : static_cast<uint16_t>(0);
                    }
                }
                if (has_mb) {
                    uint32_t *dst = reinterpret_cast<uint32_t *>(st + L.vmb);
                    if (a.al_mb && full) {
                        for (int i = lane; i < rows_here * 32; i += 32) {
                            const int r = i >> 5, pc = i & 31;
                            cp16(dst + r * 128 + 4 * pc, a.mbool + static_cast<size_t>(q0 + r) * N + t0 + 4 * pc);
                        }
                    } else {
                        for (int i = lane; i < rows_here * 128; i += 32) {
                            const int r = i >> 7, k = i & 127;
                            dst[i] = k < tval ? a.mbool[static_cast<size_t>(q0 + r) * N + t0 + k] : 0u;
                        }
                    }
                }
                if (has_mf) {
                    uint16_t *dst = reinterpret_cast<uint16_t *>(st + L.vmf);
                    const uint16_t *mf = static_cast<const uint16_t *>(a.mfloat);
                    if (a.al_mf && full) {
                        for (int i = lane; i < rows_here * 16; i += 32) {
                            const int r = i >> 4, pc = i & 15;
                            cp16(dst + r * 128 + 8 * pc, mf + static_cast<size_t>(q0 + r) * N + t0 + 8 * pc);
                        }
                    } else {
                        for (int i = lane; i < rows_here * 128; i += 32) {
                            const int r = i >> 7, k = i & 127;
                            dst[i] = k < tval ? mf[static_cast<size_t>(q0 + r) * N + t0 + k] : static_cast<uint16_t>(0);
                        }
                    }
                }
                cp_arrive_noinc(&bars->vfull[slot]);   // when this lane's cp.async copies have landed
                mbar_arrive(&bars->vfull[slot]);       // after this lane's plain stores (release)
            }
        }
        // Drain: every copy issued into this CTA's rings has landed.
        if (lane == 0) {
            for (int n = kn > NK ? kn - NK : 0; n < kn; ++n)
                if (!mbar_wait_sleep(&bars->kfull[n % NK], static_cast<uint32_t>(n / NK) & 1u, kPolls, kSleepNs)) note_abort(bars, err);
            for (int n = vn > NV ? vn - NV : 0; n < vn; ++n)
                if (!mbar_wait_sleep(&bars->vfull[n % NV], static_cast<uint32_t>(n / NV) & 1u, kPolls, kSleepNs)) note_abort(bars, err);
        }
    } else if (warp == 1 || warp == kPvWarp) {
        // --------------------------------------------------------- MMA issuers
        // Warp 1 issues the score MMAs, warp kPvWarp the PV MMAs, so that one
        // thread's waits (for decoded chunks, P, free buffers) overlap the
        // other's MMAs; each takes chunks from its own decoded ring.
        const bool is_s = warp == 1;
        if (lane == 0 && T > 0) {
            const uint32_t id_s = idesc_f16(128, RP, 0, 0, 0);
            const uint32_t id_pv = idesc_f16(128, RP, 0, 1, 0);   // A = V (MN-major), B = P (K-major)
            const uint32_t q_addr = smem_u32(smem + L.q0), d_addr = smem_u32(smem + L.d0);
            const uint32_t p_addr = smem_u32(smem + L.p0);
            const uint64_t kmaj = sw128_desc_hi(16, 1024);          // K-major operands
            // V chunks as the MN-major A operand: 64-dimension atoms one chunk apart
            const uint64_t vmn = sw128_desc_hi(kQtcChunk, 1024);
            // decoded chunks: K in slots [0, ND/2), V in [ND/2, ND), each ring in
            // order; slot and phase kept as running counters (this thread is on
            // the critical path: no divisions in its loop)
            const int NDH = ND / 2;
            int dslot[2] = {0, NDH};
            uint32_t dph[2] = {0u, 0u};
            auto take = [&](int ring, uint32_t *ca) -> bool {
                if (!wait1(bars, &bars->dfull[dslot[ring]], dph[ring], err)) return false;
                tc_fence_after();
                *ca = d_addr + static_cast<uint32_t>(dslot[ring]) * kQtcChunk;
                return true;
            };
            // the chunk after the current one (the second half of a V pair: same
            // ring pass, since a pair starts on an even slot of an even ring)
            auto take_next = [&](int ring) -> bool {
                if (!wait1(bars, &bars->dfull[dslot[ring] + 1], dph[ring], err)) return false;
                tc_fence_after();
                return true;
            };
            auto give = [&](int ring) {
                mma_commit(&bars->dempty[dslot[ring]]);
                if (++dslot[ring] == (ring + 1) * NDH) { dslot[ring] = ring * NDH; dph[ring] ^= 1u; }
            };
            const int ksg = G / 16;   // k-steps per scale group
            auto issue_s = [&](int t) -> bool {
                const int sb = t & 1;
                if (!wait1(bars, &bars->s_free[sb], ((static_cast<uint32_t>(t) >> 1) & 1u) ^ 1u, err)) return false;
                tc_fence_after();
                uint32_t acc_col = tm_s(sb), qa = q_addr;
                int kig = 0;                                // k-step within the scale group
                for (int c = 0; c < NCH; ++c) {
                    uint32_t ca;
                    if (!take(0, &ca)) return false;
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        mma_f16_ss(acc_col, sw128_desc_at(kmaj, ca + k4 * 32), sw128_desc_at(kmaj, qa + k4 * 32), id_s,
                                   kig != 0);
                        if (++kig == ksg) { kig = 0; acc_col += RP; }
                    }
                    qa += RP * 128;
                    give(0);
                }
                mma_commit(&bars->s_full[sb]);
                return true;
            };
            auto issue_pv = [&](int t) -> bool {
                if (!wait1(bars, &bars->p_full[t & 1], (static_cast<uint32_t>(t) >> 1) & 1u, err)) return false;
                tc_fence_after();
                const uint32_t pa = p_addr + (t & 1) * 4 * L.pkb;   // P_hi k-blocks, then P_lo
                // O^T[128 dims][rows] += V^T P^T per 128-dimension block: its two
                // 64-dimension chunks sit in adjacent ring slots (the V ring holds
                // an even number of chunks and a tile part starts on an even one)
                for (int mb = 0; mb < OB; ++mb) {
                    uint32_t ca;
                    if (!take(1, &ca)) return false;
                    if (NCH > 1 && !take_next(1)) return false;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t vd = sw128_desc_at(vmn, ca + kk * 2048);
                        const uint32_t pk = pa + (kk >> 2) * L.pkb + (kk & 3) * 32;
                        mma_f16_ss(tm_o + static_cast<uint32_t>(mb * RP), vd, sw128_desc_at(kmaj, pk), id_pv,
                                   (t | kk) != 0);
                        mma_f16_ss(tm_o + static_cast<uint32_t>(mb * RP), vd, sw128_desc_at(kmaj, pk + 2 * L.pkb),
                                   id_pv, 1u);
                    }
                    give(1);
                    if (NCH > 1) give(1);
                }
                mma_commit(&bars->o_done[t & 1]);
                mma_commit(&bars->p_free[t & 1]);   // P_t buffer free once PV_t is done
                return true;
            };
            bool ok = true;
            if (is_s) {
                ok = wait1(bars, &bars->q_ready, 0, err);   // Q operand staged
                tc_fence_after();
                for (int t = 0; t < T && ok; ++t) ok = issue_s(t);
            } else {
                for (int t = 0; t < T && ok; ++t) ok = issue_pv(t);
            }
            // Drain: all MMAs issued by this thread have completed.
            uint64_t *dr = is_s ? &bars->drain : &bars->drain_pv;
            mma_commit(dr);
            if (!mbar_wait_sleep(dr, 0, kPolls, kSleepNs)) note_abort(bars, err);
        }
    } else if (warp < 2 + kDecWarps) {
        // ------------------------------------------------------------ decoders
        // warps 2..5 decode K tiles into the first half of the decoded ring,
        // warps 6..9 V tiles into the second; each group runs ahead on its own
        const bool is_v = warp >= 2 + kDecGroup;
        const int dtid = tid - 64 - (is_v ? 32 * kDecGroup : 0);
        const int NDH = ND / 2;
        const int ds0 = is_v ? NDH : 0;
        int ds = ds0;                                       // ring slot and its pass parity
        uint32_t dph = 0u;
        bool ok = true;
#pragma unroll 1
        for (int t = 0; t < T && ok; ++t) {
            const int slot = is_v ? t % NV : t % NK;
            uint64_t *full = is_v ? &bars->vfull[slot] : &bars->kfull[slot];
            ok = waitw(bars, full, static_cast<uint32_t>(t / (is_v ? NV : NK)) & 1u, err);
            if (!ok) break;
            const unsigned char *words = is_v ? smem + L.v0 + slot * L.vslot + L.vw : smem + L.k0 + slot * L.kslot;
            const unsigned char *vst = smem + L.v0 + slot * L.vslot;
            const uint16_t *vs = reinterpret_cast<const uint16_t *>(vst + L.vvs);
            const uint16_t *vb = reinterpret_cast<const uint16_t *>(vst + L.vvb);
#pragma unroll 1
            for (int c = 0; c < NCH && ok; ++c) {
                ok = waitw(bars, &bars->dempty[ds], dph ^ 1u, err);
                if (!ok) break;
                decode_chunk<BITS>(reinterpret_cast<const uint32_t *>(words), WPT, c, smem + L.d0 + ds * kQtcChunk, dtid,
                                   is_v, vs, vb, NG, G, bf16);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->dfull[ds]);
                if (++ds == ds0 + NDH) { ds = ds0; dph ^= 1u; }
            }
            __syncwarp();
            if (lane == 0 && ok) mbar_arrive(is_v ? &bars->vempty[slot] : &bars->kempty[slot]);
        }
    } else {
        // -------------------------------------------- softmax and epilogue
        const int half = sw >> 2;                           // rows [half * RH, half * RH + RH)
        const int quarter = warp & 3;
        const int tl = quarter * 32 + lane;                 // token of the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const int hr0 = half * RH;
        const bool o_warp = half == 0;                      // the first half's warps own O^T (all lanes)
        auto half_sync = [&]() { asm volatile("bar.sync %0, 128;" ::"r"(1 + half) : "memory"); };
        auto all_sync = [&]() { asm volatile("bar.sync 3, 256;" ::: "memory"); };

        // ---- Q operand (f16, rows scaled by 2^-e_r) and per-row constants from
        // the rows fetched at the start
        {
            const float qs = a.scale * kLog2e;
            auto &x = qx;
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                const int r = sw + kSmWarps * i;
                const bool live = r < rows_here;
                float amax = 0.0f, gs = 0.0f;
#pragma unroll
                for (int e = 0; e < 8; ++e) { amax = fmaxf(amax, fabsf(x[i][e])); gs += x[i][e]; }
                amax = warp_max(amax);
                // 2^ex with max |q'| = max |q| * 2^-ex in [2^14, 2^15): the exponent
                // field of amax, clamped so that both 2^ex and 2^-ex are normal
                // floats (a row whose entries are all below 2^-100 scales to zeros)
                int ex = amax > 0.0f ? static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 127 - 14 : 0;
                ex = max(-100, min(100, ex));
                const float up = __uint_as_float(static_cast<uint32_t>(127 + ex) << 23);     // 2^ex
                const float down = __uint_as_float(static_cast<uint32_t>(127 - ex) << 23);   // 2^-ex
                const int lpg = G / E;                      // lanes per scale group (power of two <= 32)
                for (int m = 1; m < lpg; m <<= 1) gs += __shfl_xor_sync(0xffffffffu, gs, m);
                // the bias term in units of the row factor: sum_g b_g * 2^-e_r * sum_{d in g} q_d
                if (lane % lpg == 0) sQG[(lane * E / G) * RP + r] = live ? gs * down : 0.0f;
                if (lane == 0) sF[r] = live ? qs * up : 0.0f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if (e >= E) break;
                    const int d = lane * E + e;
                    const int pos = BITS == 4 ? ((d & ~7) | pos4(d & 7)) : d;
                    const int blk = pos >> 6, pc = (pos & 63) >> 3;
                    *reinterpret_cast<__half *>(smem + L.q0 + blk * RP * 128 + r * 128 + ((pc ^ (r & 7)) << 4) +
                                                (pos & 7) * 2) = __float2half_rn(x[i][e] * down);
                }
            }
            // draft tree over the last tree_ql tokens: node bitsets, by the first warp
            if (sw == 0 && a.tree_ql > 0) {
                const uint32_t anc = quant_tree_ancestors(tree_up, a.tree_ql);
                if (lane < a.tree_ql) sTree[lane] = anc;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->q_ready);
        }
        bool ok = waitw(bars, &bars->q_ready, 0, err);      // every warp's rows (sF, sQG, sTree)
        const int tree_lo = N - a.tree_ql;

        float lsum[RH];
#pragma unroll
        for (int r = 0; r < RH; ++r) lsum[r] = 0.0f;
        float m_row = -INFINITY;                            // running max (log2 units) of row hr0 + lane % RH
#pragma unroll 1
        for (int t = 0; t < T; ++t) {
            const int sb = t & 1;
            const int vslot = t % NV;
            const int tok = (j0 + t) * 128 + tl;
            const bool tok_ok = tok >= a.t_lo && tok < N;
            ok = ok && waitw(bars, &bars->vfull[vslot], static_cast<uint32_t>(t / NV) & 1u, err);
            ok = ok && waitw(bars, &bars->s_full[sb], (static_cast<uint32_t>(t) >> 1) & 1u, err);
            tc_fence_after();
            const unsigned char *st = smem + L.v0 + vslot * L.vslot;
            const uint16_t *ks = reinterpret_cast<const uint16_t *>(st + L.vks);
            const uint16_t *kb = reinterpret_cast<const uint16_t *>(st + L.vkb);
            float acc[RH];   // sum_g s_g S^T_g + b_g * 2^-e_r * sum_{d in g} q_d
#pragma unroll
            for (int r = 0; r < RH; ++r) acc[r] = 0.0f;
            if (ok) {
#pragma unroll 1
                for (int g = 0; g < NG; ++g) {
                    uint32_t d[RH];
                    tmem_ldn<RH>(tm_s(sb) + lane_off + static_cast<uint32_t>(g * RP + hr0), d);
                    tmem_wait_ld();
                    const float s = t2f(ks[tl * NG + g], bf16), b = t2f(kb[tl * NG + g], bf16);
                    const float *qg = sQG + g * RP + hr0;
#pragma unroll
                    for (int r = 0; r < RH; ++r) acc[r] = fmaf(s, __uint_as_float(d[r]), fmaf(b, qg[r], acc[r]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0 && ok) mbar_arrive(&bars->s_free[sb]);   // S_t read out of TMEM
            float (&lg)[RH] = acc;   // logits (log2 units), in place
            const bool live_tok = ok && tok_ok;
#pragma unroll
            for (int r = 0; r < RH; ++r) lg[r] = (live_tok && hr0 + r < rows_here) ? acc[r] * sF[hr0 + r] : -INFINITY;
            if (has_mf) {
                const uint16_t *mf = reinterpret_cast<const uint16_t *>(st + L.vmf) + tl;
#pragma unroll
                for (int r = 0; r < RH; ++r)
                    if (hr0 + r < rows_here) lg[r] = fmaf(kLog2e, t2f(mf[(hr0 + r) * 128], bf16), lg[r]);
            }
            if (has_mb) {
                const uint32_t *mb = reinterpret_cast<const uint32_t *>(st + L.vmb) + tl;
#pragma unroll
                for (int r = 0; r < RH; ++r)
                    if (hr0 + r < rows_here && mb[(hr0 + r) * 128] == 0u) lg[r] = -INFINITY;
            }
            if (a.tree_ql > 0 && tok >= tree_lo && tok < N) {
                // a tree position: row q attends it if it is node q % tree_ql or one of its ancestors
                const int jt = tok - tree_lo;
#pragma unroll
                for (int r = 0; r < RH; ++r)
                    if (!((sTree[(q0 + hr0 + r) % a.tree_ql] >> jt) & 1u)) lg[r] = -INFINITY;
            }
            __syncwarp();
            if (lane == 0 && ok) mbar_arrive(&bars->vempty[vslot]);   // scales and masks read

            // row maxima of the tile: warp reduce-scatter, then the half's four warps
            float tmp[RH];
#pragma unroll
            for (int r = 0; r < RH; ++r) tmp[r] = lg[r];
            float wm = reduce_scatter<RH, true>(tmp, lane);
#pragma unroll
            for (int m = RH; m < 32; m <<= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, m));
            float *mx = sMax + (sb * 2 + half) * 128;
            mx[quarter * 32 + lane] = wm;
            half_sync();
            const float tmax = fmaxf(fmaxf(mx[lane], mx[32 + lane]), fmaxf(mx[64 + lane], mx[96 + lane]));
            float alpha = 1.0f;
            if (tmax > m_row + kSlack) {
                alpha = m_row == -INFINITY ? 0.0f : ex2(m_row - tmax);
                m_row = tmax;
            }
            const bool need = __any_sync(0xffffffffu, alpha != 1.0f);   // same in the half's four warps
            if (need) {
#pragma unroll
                for (int r = 0; r < RH; ++r) lsum[r] *= __shfl_sync(0xffffffffu, alpha, r);
            }
            // the P buffer of this tile is free once PV of tile t - 2 is done
            ok = ok && waitw(bars, &bars->p_free[sb], ((static_cast<uint32_t>(t) >> 1) & 1u) ^ 1u, err);
            if (need && t > 0) {
                // this half's rows moved their max: the half's four warps rescale
                // the rows' columns of O^T (their lanes) once PV of the previous
                // tile is done; the other half's columns are its own business
                ok = ok && waitw(bars, &bars->o_done[(t - 1) & 1], (static_cast<uint32_t>(t - 1) >> 1) & 1u, err);
                tc_fence_after();
                if (ok) {
#pragma unroll 1
                    for (int mb = 0; mb < OB; ++mb) {
                        const uint32_t col = tm_o + lane_off + static_cast<uint32_t>(mb * RP + hr0);
                        uint32_t v[RH];
                        tmem_ldn<RH>(col, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int r = 0; r < RH; ++r)
                            v[r] = __float_as_uint(__uint_as_float(v[r]) * __shfl_sync(0xffffffffu, alpha, r));
                        tmem_stn<RH>(col, v);
                    }
                    tmem_wait_st();
                }
            }
            // P as two f16 terms, P_hi = rn(P) and P_lo = rn(P - P_hi) (the
            // difference is exact in f32), in the P_hi and P_lo k-blocks of the
            // buffer: one f16 P would move the output by up to 2^-11 of the
            // spread of the attended V values, the pair by less than 2^-22.
            // The row sums add P in f32.
            unsigned char *pb = smem + L.p0 + sb * 4 * L.pkb + (tl >> 6) * L.pkb;
            const int tc = tl & 63;
#pragma unroll
            for (int r = 0; r < RH; ++r) {
                const int row = hr0 + r;
                const float m = __shfl_sync(0xffffffffu, m_row, r);
                const float pf = ex2(lg[r] - (m == -INFINITY ? 0.0f : m));
                const __half ph = __float2half_rn(pf);
                const __half pl = __float2half_rn(pf - __half2float(ph));
                lsum[r] += pf;
                if (row < rows_here) {
                    const int off = row * 128 + (((tc >> 3) ^ (row & 7)) << 4) + (tc & 7) * 2;
                    *reinterpret_cast<__half *>(pb + off) = ph;
                    *reinterpret_cast<__half *>(pb + 2 * L.pkb + off) = pl;
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0 && ok) mbar_arrive(&bars->p_full[sb]);
        }
        pdl_launch_dependents();   // the merge may start launching; it waits for this grid to finish
        if (T > 0 && o_warp) {
            ok = ok && waitw(bars, &bars->o_done[(T - 1) & 1], (static_cast<uint32_t>(T - 1) >> 1) & 1u, err);
            tc_fence_after();
        }
        // row sums over the tokens of the half's four warps; final row maxima
        float ls = reduce_scatter<RH, false>(lsum, lane);
#pragma unroll
        for (int m = RH; m < 32; m <<= 1) ls += __shfl_xor_sync(0xffffffffu, ls, m);
        sSum[(half * 4 + quarter) * 32 + lane] = ls;
        if (quarter == 0 && lane < RH) sMrow[hr0 + lane] = m_row;
        all_sync();
        if (o_warp && ok) {
            // the first half's four warps: lane = a dimension position of each
            // 128-dimension block (TMEM lane quarter * 32 + lane), column = row
            const int pos = quarter * 32 + lane;             // 0..127
            // dimension held at that position (4-bit words decode to positions 0,4,1,5,2,6,3,7)
            const int p8 = pos & 7;
            const int dpos = (pos & ~7) | (BITS == 4 ? ((p8 >> 1) | ((p8 & 1) << 2)) : p8);
            // output factor of row r: 1 for a partial, else 1 / (l + sink term)
            auto row_factor = [&](int r) -> float {
                if (a.nwg > 1) return 1.0f;
                const float *sh = sSum + (r / RH) * 128 + (r % RH);
                const float l_tot = (sh[0] + sh[32]) + (sh[64] + sh[96]);
                const float m_fin = sMrow[r];
                float cf = 1.0f, sf = l_tot;
                if (a.has_sinks) {
                    const float sk = kLog2e * __ldg(a.sinks + ((q0 + r) % a.nQ));
                    const float mx = fmaxf(m_fin, sk);
                    cf = m_fin == -INFINITY ? 0.0f : ex2(m_fin - mx);
                    sf = l_tot * cf + ex2(sk - mx);
                }
                return sf > 0.0f ? cf / sf : 0.0f;
            };
#pragma unroll 1
            for (int mb = 0; mb < OB; ++mb) {
                uint32_t v[RP];
                if (T > 0) {
                    tmem_ldn<RP>(tm_o + lane_off + static_cast<uint32_t>(mb * RP), v);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int j = 0; j < RP; ++j) v[j] = 0u;
                }
                const int d = mb * 128 + dpos;
                if (d >= DIM) continue;
#pragma unroll
                for (int r = 0; r < RR; ++r) {
                    if (r >= rows_here) break;
                    const float o = __uint_as_float(v[r]) * row_factor(r);
                    const size_t idx = static_cast<size_t>(q0 + r) * DIM + d;
                    if (a.nwg > 1) a.part_o[static_cast<size_t>(split) * a.rows * DIM + idx] = o;
                    else if (a.out_f32) static_cast<float *>(a.out)[idx] = o;
                    else if (bf16) static_cast<__nv_bfloat16 *>(a.out)[idx] = __float2bfloat16_rn(o);
                    else static_cast<__half *>(a.out)[idx] = __float2half_rn(o);
                }
            }
            if (a.nwg > 1 && quarter == 0 && lane < rows_here) {
                const float *sh = sSum + (lane / RH) * 128 + (lane % RH);
                reinterpret_cast<float2 *>(a.part_ml)[static_cast<size_t>(split) * a.rows + q0 + lane] =
                    make_float2((sh[0] + sh[32]) + (sh[64] + sh[96]), sMrow[lane]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, static_cast<uint32_t>(a.tc_cols));
    }
}

template <int BITS, int RR>
cudaError_t launch_rr(const QuantArgs &a, size_t smem, cudaStream_t s) {
    auto kern = quant_tc_kernel<BITS, RR>;
    static unsigned long long done = 0;
    cudaError_t e = set_smem_limit_once(kern, kQuantMaxSmem, &done);
    if (e != cudaSuccess) return e;
    kern<<<dim3(a.nwg, a.kv_rows * a.n_rb), kThreads, smem, s>>>(a);
    count_launch();
    return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_bits(const QuantArgs &a, size_t smem, cudaStream_t s) {
    switch (a.rp) {
        case 4: return launch_rr<BITS, 4>(a, smem, s);
        case 8: return launch_rr<BITS, 8>(a, smem, s);
        case 16: return launch_rr<BITS, 16>(a, smem, s);
        case 32: return launch_rr<BITS, 32>(a, smem, s);
        default: return cudaErrorInvalidValue;
    }
}

template <int BITS, int RR>
int occupancy_rr(size_t smem) {
    auto kern = quant_tc_kernel<BITS, RR>;
    static unsigned long long done = 0;
    if (set_smem_limit_once(kern, kQuantMaxSmem, &done) != cudaSuccess) { cudaGetLastError(); return 0; }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

template <int BITS>
int occupancy_bits(int rp, size_t smem) {
    return rp <= 4 ? occupancy_rr<BITS, 4>(smem) : rp <= 8 ? occupancy_rr<BITS, 8>(smem)
         : rp <= 16 ? occupancy_rr<BITS, 16>(smem) : occupancy_rr<BITS, 32>(smem);
}

}  // namespace qtc
}  // namespace ta
