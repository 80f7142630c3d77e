// Tensor-core (tcgen05) tree-verify attention main pass for f16 / bf16 K/V.
//
// Semantics are those of mlx-native tree_attention.metal (tree_attention_impl):
// logit = fma(qk, scale, mask); a 32-key chunk whose mask cells are all
// <= -65504 for a row contributes nothing to that row; online softmax with a
// running max M and sum S; partial (O, S, M) per split, merged by the reduce
// pass (or normalized here when there is a single split).  The Metal kernel
// walks one query row per threadgroup with CUDA-core-style dot products; here
// all query rows of a KV head are one dense contraction for the tensor core.
//
// One CTA = (split, 128-row tile x O-column half, KV head).  Rows r of KV head
// k are (head k*g + r / L, query r % L), contiguous in the 16-bit Q copy.
//   warp 0     : TMA producer - the Q tile once, then K and V slabs
//                ([128 keys x 64 cols] 16-bit, 128-byte swizzle) through a ring
//                of 16 KB stages, in the order the MMA warp consumes them
//                (K_0, K_1, V_0, K_2, V_1, ...).  A split owns a contiguous
//                range of 32-key chunks; a tile holds its next 4 live chunks
//                (dead chunks are never loaded); empty slots and keys past
//                kv_seq_len are loaded out of bounds, i.e. as zeros.
//   warp 1     : TMEM owner and MMA issuer: S_t = Q K_t^T (M 128, N 128, f32 in
//                TMEM, double buffered) and O += P_t V_t (M 128, N = 64 per V
//                slab, up to 256 over slabs in consecutive ring slots; P read
//                from TMEM where the softmax left it over S_t, V MN-major); the
//                QK^T and PV MMAs are issued by two threads (warps 1 and 11)
//                and S_t+2 reuses the buffer of S_t once PV_t has completed.
//   warps 2..9 : two warps per TMEM lane quarter: mask + scale, online softmax
//                with lazy rescaling (M only moves when a row max exceeds it by
//                more than e^8, so O in TMEM is rarely touched), P back into
//                TMEM as two 16-bit terms P = P_hi + P_lo, epilogue from TMEM.
//   warp 10    : second TMA producer of a CTA pair (alternate ring loads).
// P in two terms: the tensor core takes 16-bit operands, and a single 16-bit
// P carries a relative rounding error of up to 2^-8 (bf16) or 2^-11 (f16),
// which moves the output by up to that fraction of the spread of the attended
// V rows - above the 2e-3 tolerance on a peaked softmax.  P_hi = rn16(P) and
// P_lo = rn16(P - P_hi) (the difference is exact in f32) leave a relative
// error below 2^-16 (bf16) or 2^-22 (f16); PV runs once per term.
// Every mbarrier wait is bounded; on a timeout the CTA sets the workspace
// error word, drains its outstanding copies and MMAs, frees TMEM and exits.
// Every CTA loads its own K/V slabs (a row tile's second read of a slab is
// usually an L2 hit).
#include "sm100_ptx.cuh"
#include "ta_internal.cuh"

namespace ta {

namespace {

using namespace sm100;

// warp 0: producer 0, warp 1: QK issuer + TMEM owner, warps 2-9: softmax,
// warp 10: producer 1, warp 11: PV issuer
constexpr int kTcWarps = 12;
constexpr int kPvWarp = 11;
constexpr int kProd1Warp = 10;
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kSlab = 16384;                 // [128 rows][64 x 16-bit], 128-byte swizzled
constexpr uint32_t kWaitIters = 1u << 22;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleSlack2 = 8.0f * kLog2e;   // in log2 units: P <= e^8 = 2981 fits f16 and bf16

// PAIR = false: one CTA per 128-row tile (cta_group::1), ring slots of 16 KB
// ([128 keys x 64 cols]).  PAIR = true: a CTA pair (cta_group::2) covers two
// row tiles with M = 256 MMAs, and each CTA loads half of every operand tile:
// 64 of a key tile's 128 keys for QK^T, half of the O columns of V for PV;
// ring slots of 8 KB ([64 keys x 64 cols]).
template <int D, bool PAIR>
struct TcCfg {
    static constexpr int DV = D < 256 ? D : 256;     // O columns per CTA (its rows' share of O)
    static constexpr int NSK = D / 64;               // K slots per key tile
    static constexpr int NSV = DV / 64;              // V slots per key tile
    static constexpr int SLOT = PAIR ? 8192 : kSlab; // bytes of a ring slot
    // Ring depth.  Every key tile advances the ring by NSK + NSV slots and a V
    // group starts NSV-aligned, so with these depths a tile's V slots sit in
    // runs of consecutive slots (single CTA: D 128, 256 one run, D 512 slots
    // 4, 5 | 0, 1; pair: always one run) that one PV instruction covers.
    static constexpr int STAGES = PAIR ? (D == 512 ? 12 : (D == 256 ? 16 : 24))
                                       : (D == 512 ? 6 : (D == 256 ? 8 : 12));
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_RING = OFF_Q + NSK * kSlab;
    static constexpr int OFF_BAR = OFF_RING + STAGES * SLOT;
    static constexpr int SMEM = OFF_BAR + 3072;      // the dynamic base must be 1024-aligned
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(128 * (DV + 4) * 4 + 128 * 8 <= OFF_BAR, "epilogue staging fits below the barriers");
};

constexpr int kMaxStages = 24;

struct Bars {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t q_full;
    uint64_t s_full[2];
    uint64_t p_full;
    uint64_t s_free[2];   // PV of tiles t = b (mod 2) done: S buffer b may be overwritten
    uint64_t drain_pv;
    uint64_t o_done[2];   // PV of tiles t = b (mod 2) done
    uint64_t drain;
    uint64_t peer_done[2];   // pair: the peer's producer p has published how far it issued
    uint32_t tmem_base;
    uint32_t peer_issued[2]; // pair: 1 + index of the last ring load the peer's producer p issued
    volatile int abort_flag;
    float xrow[2][2][128];   // per-row values exchanged by the two warps of a TMEM quarter
};
static_assert(sizeof(Bars) <= 3072, "barrier area");

// Walk of the live (not dead) 32-key chunks of the chunk-index range
// [begin, end) of this split, in order.  Warp-collective: all lanes call it
// together and hold the same state.
struct ChunkWalk {
    const uint8_t *cls;
    int base, end, my_cls;      // my_cls: class of chunk base + lane
    uint32_t pending;

    __device__ void load(int b) {
        const int c = b + static_cast<int>(threadIdx.x & 31);
        my_cls = c < end ? cls[c] : kChunkDead;
        pending = __ballot_sync(0xffffffffu, my_cls != kChunkDead);
    }
    __device__ void init(const uint8_t *c, int begin, int end_) {
        cls = c;
        base = begin;
        end = end_;
        pending = 0u;
        my_cls = kChunkDead;
        if (base < end) load(base);
    }
    // Next live chunk index (and its class), or -1 when the range is exhausted.
    __device__ int next(int *cl) {
        while (pending == 0) {
            base += 32;
            if (base >= end) return -1;
            load(base);
        }
        const int bit = __ffs(pending) - 1;
        pending &= pending - 1;
        *cl = __shfl_sync(0xffffffffu, my_cls, bit);
        return base + bit;
    }
};

// Chunk-index range of a split: whole 4-chunk tiles, ceil(tiles / nwg) each.
__device__ __forceinline__ void split_range(int n_chunks, int nwg, int split, int *begin, int *end) {
    const int tiles = (n_chunks + 3) / 4;
    const int cps = ((tiles + nwg - 1) / nwg) * 4;
    *begin = min(n_chunks, split * cps);
    *end = min(n_chunks, *begin + cps);
}

// Number of 4-chunk key tiles of the split's live chunks (warp-collective).
__device__ __forceinline__ int count_tiles(const uint8_t *cls, int begin, int end) {
    const int lane = threadIdx.x & 31;
    int n = 0;
    for (int b = begin; b < end; b += 32)
        n += __popc(__ballot_sync(0xffffffffu, b + lane < end && cls[b + lane] != kChunkDead));
    return (n + 3) / 4;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Abort: flag this CTA (and, in a pair, the peer: peer_flag is the
// shared::cluster address of its flag, 0 for none) and record the first code.
__device__ __forceinline__ void note_abort(Bars *b, int *err, int code, uint32_t peer_flag) {
    b->abort_flag = 1;
    if (peer_flag != 0u) st_dsmem_u32(peer_flag, 1u);
    atomicCAS(err, 0, code);
}

// Suspend-time hint (ns) of the waits of the producers and MMA issuers, whose
// wake-up latency is on the ring's critical path; the softmax warps use 1 us.
constexpr uint32_t kPipeHintNs = 1000;

__device__ __forceinline__ bool wait_or_abort(Bars *b, uint64_t *bar, uint32_t parity, int *err, int code,
                                              uint32_t peer_flag, uint32_t hint_ns = 1000) {
    if (b->abort_flag) return false;
    // a waiting warp sleeps on the barrier (taking no issue slots from the
    // other warps), at most about 2 s in all
    if (mbar_try_wait(bar, parity) || mbar_wait_sleep(bar, parity, (1u << 21) * (1000u / hint_ns), hint_ns))
        return true;
    note_abort(b, err, code, peer_flag);
    return false;
}

// As wait_or_abort, for a barrier that threads of the peer CTA arrive on
// (acquire at cluster scope).
__device__ __forceinline__ bool wait_or_abort_cluster(Bars *b, uint64_t *bar, uint32_t parity, int *err, int code,
                                                      uint32_t peer_flag, uint32_t hint_ns = 1000) {
    if (b->abort_flag) return false;
    for (uint32_t i = 0; i < (1u << 21) * (1000u / hint_ns); ++i)
        if (mbar_try_wait_cluster(bar, parity, hint_ns)) return true;
    note_abort(b, err, code, peer_flag);
    return false;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
    if (bf16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    }
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ float lo16(uint32_t u, bool bf16) {
    if (bf16) return __uint_as_float(u << 16);
    return __half2float(__ushort_as_half(static_cast<unsigned short>(u & 0xffffu)));
}
__device__ __forceinline__ float hi16(uint32_t u, bool bf16) {
    if (bf16) return __uint_as_float(u & 0xffff0000u);
    return __half2float(__ushort_as_half(static_cast<unsigned short>(u >> 16)));
}

template <int D, bool BF16, bool IMPLICIT, bool PAIR>
__global__ void __launch_bounds__(kTcThreads, 1) tree_tc_kernel(const TreeArgs a, const __grid_constant__ TcMaps maps) {
    using Cfg = TcCfg<D, PAIR>;
    constexpr int DV = Cfg::DV, NSK = Cfg::NSK, NSV = Cfg::NSV, ST = Cfg::STAGES, SLOT = Cfg::SLOT;
    static_assert(ST <= kMaxStages, "ring depth");
    constexpr int SROW = DV + 4;                        // floats per staged O row
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 128-byte-swizzled TMA / MMA tiles need a 1024-byte-aligned base; every
    // CTA has the same base, so a misaligned one stops all of them before any
    // barrier or allocation.
    if ((smem_u32(smem_raw) & 1023u) != 0) {
        if (threadIdx.x == 0) atomicCAS(a.err, 0, 11);
        return;
    }
    unsigned char *sm = smem_raw;
    unsigned char *sQ = sm + Cfg::OFF_Q;
    unsigned char *sRing = sm + Cfg::OFF_RING;
    Bars *bars = reinterpret_cast<Bars *>(sm + Cfg::OFF_BAR);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Grid.  Single CTA: x = split, y = O half * row tiles + row tile.  Pair:
    // x = 2 * (pair of row tiles) + member, y = split * O halves + O half; the
    // cluster is the pair (cluster ranks 2k, 2k + 1), member 0 the leader that
    // issues the MMAs.  z = KV head.  Flattened pairs: x = member, y = group *
    // O halves + O half, z = 0; the group's work segments name the KV head and
    // row tiles.
    constexpr int kHalves = D / DV;
    const int n_ct = tree_tc_row_ctas(a.R, D);         // row tiles
    const int member = PAIR ? static_cast<int>(cluster_ctarank() & 1u) : 0;
    const bool leader = member == 0;
    const bool flat = PAIR && a.flat_groups > 0;
    const int split = flat ? 0 : (PAIR ? static_cast<int>(blockIdx.y) / kHalves : static_cast<int>(blockIdx.x));
    const int os = PAIR ? static_cast<int>(blockIdx.y) % kHalves : static_cast<int>(blockIdx.y) / n_ct;
    const int RT = (a.R + n_ct - 1) / n_ct;            // rows per tile
    // the current work segment's KV head and row tile (set per segment below)
    int kh = blockIdx.z;
    int rt = PAIR ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.y) % n_ct;
    int rows_here = min(RT, a.R - rt * RT);
    int *err = a.err;
    // Cluster (single CTA: cx x 1): consecutive splits of one (row tile, O
    // half, KV head) whose partials are merged in the cluster over DSMEM.
    // Pair: the cluster is the pair and splits are never merged in it.
    const int cx = PAIR ? 1 : static_cast<int>(cluster_nctaid_x());
    const int cxi = PAIR ? 0 : static_cast<int>(cluster_ctaid_x());
    // shared::cluster addresses: the leader's barriers (pair), the peer's abort flag
    const uint32_t lead_rank = PAIR ? (cluster_ctarank() & ~1u) : 0u;
    const uint32_t peer_rank = PAIR ? (cluster_ctarank() ^ 1u) : 0u;
    const uint32_t peer_flag =
        PAIR ? mapa_shared(smem_u32(const_cast<int *>(&bars->abort_flag)), peer_rank) : 0u;
    auto at_leader = [&](const void *p) -> uint32_t { return mapa_shared(smem_u32(p), lead_rank); };
    auto at_peer = [&](const void *p) -> uint32_t { return mapa_shared(smem_u32(p), peer_rank); };

    if (tid == 0) {
        for (int i = 0; i < ST; ++i) { mbar_init(&bars->full[i], 1); mbar_init(&bars->empty[i], 1); }
        mbar_init(&bars->q_full, 1);
        for (int i = 0; i < 2; ++i) { mbar_init(&bars->s_full[i], 1); mbar_init(&bars->s_free[i], 1); }
        mbar_init(&bars->drain_pv, 1);
        mbar_init(&bars->p_full, PAIR ? 16 : 8);       // the softmax warps (of both CTAs of a pair)
        mbar_init(&bars->o_done[0], 1);
        mbar_init(&bars->o_done[1], 1);
        mbar_init(&bars->drain, 1);
        mbar_init(&bars->peer_done[0], 1);
        mbar_init(&bars->peer_done[1], 1);
        bars->peer_issued[0] = bars->peer_issued[1] = 0u;
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(&bars->tmem_base, 512);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&bars->tmem_base, 512);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    cluster_sync();                                     // peers' barriers exist before any remote access
    tc_fence_after();
    pdl_wait();                                         // chunk classes and Q copy are ready
    const uint32_t tmem = bars->tmem_base;
    const uint32_t tm_s[2] = {tmem, tmem + 128};
    const uint32_t tm_o = tmem + 256;

    // Work segments of this CTA: (KV head, row tile, chunk range, partial
    // slot, live tiles).  Uniform splits: one segment.  Flattened pairs: the
    // group's range of (unit, key tile) positions, in at most two units; a
    // segment ending its unit also marks the unit's unused slots empty.  The
    // segments' tiles form one sequence through the ring and the barriers.
    int nseg = 1;
    int sg_kh[2], sg_rt[2], sg_cb[2], sg_ce[2], sg_slot[2], sg_T[2], sg_used[2];
    bool sg_last[2];
    if (flat) {
        const int G = a.flat_groups, grp = static_cast<int>(blockIdx.y) / kHalves;
        const int np = n_ct / 2, tpu = (a.n_chunks + 3) / 4;
        const long long W = static_cast<long long>(a.Hk) * np * tpu;
        const long long p1 = flat_start(grp + 1, W, G);
        nseg = 0;
        for (long long P = flat_start(grp, W, G); P < p1 && nseg < 2; ++nseg) {
            const int u = static_cast<int>(P / tpu);
            const long long ub = static_cast<long long>(u) * tpu, e = min(p1, ub + tpu);
            sg_kh[nseg] = u / np;
            sg_rt[nseg] = 2 * (u % np) + member;
            sg_cb[nseg] = static_cast<int>(P - ub) * 4;
            sg_ce[nseg] = min(a.n_chunks, static_cast<int>(e - ub) * 4);
            sg_slot[nseg] = grp - flat_group_of(ub, W, G);
            sg_used[nseg] = flat_unit_slots(u, tpu, W, G);
            sg_last[nseg] = e == ub + tpu;
            P = e;
        }
    } else {
        sg_kh[0] = kh;
        sg_rt[0] = rt;
        split_range(a.n_chunks, a.nwg, split, &sg_cb[0], &sg_ce[0]);
        sg_slot[0] = split;
        sg_used[0] = a.nwg;
        sg_last[0] = false;
    }
    int T = 0;                                          // tiles of all segments
    for (int i = 0; i < nseg; ++i) {
        sg_T[i] = count_tiles(a.cls, sg_cb[i], sg_ce[i]);
        T += sg_T[i];
    }
    auto enter_segment = [&](int i) {
        kh = sg_kh[i];
        rt = sg_rt[i];
        rows_here = min(RT, a.R - rt * RT);
    };
    enter_segment(0);
    const int n_pad = ((a.N + 31) / 32) * 32;          // a key row that is out of bounds

    if (warp == 0 || warp == kProd1Warp) {
        // ----------------------------------------------------------- producers
        // Pair: two producer warps issue alternate ring loads (global load
        // index n: producer n % 2): one thread issuing 8 KB copies back to back
        // is limited by the issue time of each copy, two reach the rate HBM can
        // feed an SM.  Both walk the whole sequence.  Single CTA: warp 0 issues
        // every load (measured faster there; warp kProd1Warp only idles).
        const int prod = warp == 0 ? 0 : 1;
        auto mine = [&](int n) { return PAIR ? (n & 1) == prod : prod == 0; };
        ChunkWalk walk;
        int issued = 0;                                 // ring loads of the sequence so far (both producers)
        int mine_end = 0;                               // 1 + index of the last load this producer issued
        // Single CTA: a slab's 4 chunks as four 32-key boxes (a missing chunk
        // loads zeros from past kv_seq_len); one 128-key or two 64-key boxes
        // for consecutive chunks measured slower here.
        auto load_slabs = [&](const int (&chunk)[4], int nslab, int x0, bool is_v) -> bool {
            const CUtensorMap *m32 = is_v ? &maps.v : &maps.k;
            for (int s = 0; s < nslab; ++s, ++issued) {
                if (!mine(issued)) continue;
                const int slot = issued % ST;
                const uint32_t pass = static_cast<uint32_t>(issued / ST);
                bool ok = true;
                if (lane == 0) {
                    ok = wait_or_abort(bars, &bars->empty[slot], (pass & 1u) ^ 1u, err, 1, 0u, kPipeHintNs);
                    if (ok) {
                        mbar_arrive_expect_tx(&bars->full[slot], kSlab);
                        unsigned char *dst = sRing + slot * SLOT;
                        const int xx = x0 + s * 64;
                        for (int c = 0; c < 4; ++c)
                            tma_load_3d(dst + c * 4096, m32, &bars->full[slot], xx,
                                        chunk[c] >= 0 ? chunk[c] * 32 : n_pad, kh);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) return false;
                mine_end = issued + 1;
            }
            return true;
        };
        // Pair: one slot = the 64 keys of chunks c0, c1 (one 64-key box when they
        // are consecutive, else two 32-key boxes; a missing chunk loads zeros)
        // x 64 columns from x0, into this CTA's slot; the copy completes on the
        // leader's full barrier, which expects both CTAs' 8 KB.
        auto load_unit = [&](const CUtensorMap *map, const CUtensorMap *map64, int c0, int c1, int x0) -> bool {
            const int n = issued++;
            if ((n & 1) != prod) return true;
            const int slot = n % ST;
            const uint32_t pass = static_cast<uint32_t>(n / ST);
            bool ok = true;
            if (lane == 0) {
                ok = wait_or_abort(bars, &bars->empty[slot], (pass & 1u) ^ 1u, err, 1, peer_flag, kPipeHintNs);
                if (ok) {
                    if (leader) mbar_arrive_expect_tx(&bars->full[slot], 2 * SLOT);
                    unsigned char *dst = sRing + slot * SLOT;
                    const uint32_t fb = at_leader(&bars->full[slot]);
                    if (c0 >= 0 && c1 == c0 + 1) {
                        tma_load_3d_pair(dst, map64, fb, x0, c0 * 32, kh);
                    } else {
                        tma_load_3d_pair(dst, map, fb, x0, c0 >= 0 ? c0 * 32 : n_pad, kh);
                        tma_load_3d_pair(dst + 4096, map, fb, x0, c1 >= 0 ? c1 * 32 : n_pad, kh);
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (ok) mine_end = n + 1;
            return ok;
        };
        // Pair: K of a tile = NSK slots of this CTA's two chunks (its half of
        // the key columns of S); V = NSV slots, sub-slab j of this CTA's half
        // of the O columns in slots 2j (keys 0-63) and 2j + 1 (keys 64-127).
        auto load_k_pair = [&](const int (&chunk)[4]) -> bool {
            for (int s = 0; s < NSK; ++s)
                if (!load_unit(&maps.k, &maps.k64, chunk[2 * member], chunk[2 * member + 1], s * 64)) return false;
            return true;
        };
        auto load_v_pair = [&](const int (&chunk)[4]) -> bool {
            const int x0 = os * DV + member * (DV / 2);
            for (int j = 0; j < NSV; ++j)
                if (!load_unit(&maps.v, &maps.v64, chunk[2 * (j & 1)], chunk[2 * (j & 1) + 1], x0 + (j >> 1) * 64))
                    return false;
            return true;
        };
        bool ok = true;
        int q_loads = 0, tg0 = 0;                       // Q tiles loaded; tiles of earlier segments
        if (T > 0 && lane == 0 && prod == 0) {
            tma_prefetch_desc(&maps.k);
            tma_prefetch_desc(&maps.v);
            tma_prefetch_desc(&maps.k64);
            tma_prefetch_desc(&maps.v64);
        }
        for (int sgi = 0; sgi < nseg && ok; ++sgi) {
            const int Ts = sg_T[sgi];
            if (Ts == 0) continue;
            enter_segment(sgi);
            walk.init(a.cls, sg_cb[sgi], sg_ce[sgi]);
            if (lane == 0 && prod == 0) {
                // a later segment's Q tile replaces the earlier one once the
                // last QK^T MMAs of the earlier segment are done
                if (q_loads > 0)
                    ok = wait_or_abort(bars, &bars->s_full[(tg0 - 1) & 1],
                                       static_cast<uint32_t>((tg0 - 1) >> 1) & 1u, err, 14, peer_flag);
                if (ok) {
                    if constexpr (PAIR) {
                        if (leader) mbar_arrive_expect_tx(&bars->q_full, 2 * NSK * kSlab);
                        const uint32_t qb = at_leader(&bars->q_full);
                        for (int s = 0; s < NSK; ++s)
                            tma_load_2d_pair(sQ + s * kSlab, &maps.q16, qb, s * 64, kh * a.R + rt * RT);
                    } else {
                        mbar_arrive_expect_tx(&bars->q_full, NSK * kSlab);
                        for (int s = 0; s < NSK; ++s)
                            tma_load_2d(sQ + s * kSlab, &maps.q16, &bars->q_full, s * 64, kh * a.R + rt * RT);
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            ++q_loads;
            int cur[4], nxt[4], cl_unused;
            for (int c = 0; c < 4; ++c) nxt[c] = walk.next(&cl_unused);
            if (ok) ok = PAIR ? load_k_pair(nxt) : load_slabs(nxt, NSK, 0, false);
            for (int t = 0; t < Ts && ok; ++t) {
                for (int c = 0; c < 4; ++c) cur[c] = nxt[c];
                if (t + 1 < Ts) {
                    for (int c = 0; c < 4; ++c) nxt[c] = walk.next(&cl_unused);
                    ok = PAIR ? load_k_pair(nxt) : load_slabs(nxt, NSK, 0, false);
                }
                if (ok) ok = PAIR ? load_v_pair(cur) : load_slabs(cur, NSV, os * DV, true);
            }
            tg0 += Ts;
        }
        // Drain: every copy this producer issued into this CTA's ring has
        // landed and the MMAs have released the last use of each of its slots,
        // so nothing still targets this CTA's shared memory when it exits.  In
        // a pair the copies complete on the leader's barriers: each peer
        // producer publishes how far it issued and the leader's producer of the
        // same parity waits for every slot of that parity either CTA filled
        // (standing in, with complete_tx / expect_tx, for the bytes of a load
        // only one of them issued after an abort); the final cluster barrier
        // keeps the peer alive until then.
        if (lane == 0 && T > 0) {
            auto drain_from = [&](int end) { return end > ST ? end - ST : 0; };
            if constexpr (PAIR) {
                if (!leader) {
                    st_dsmem_u32(at_leader(&bars->peer_issued[prod]), static_cast<uint32_t>(mine_end));
                    mbar_arrive_cluster(at_leader(&bars->peer_done[prod]));
                } else {
                    int ip = mine_end;
                    bool got = false;
                    for (uint32_t i = 0; i < (1u << 21) && !got; ++i)
                        got = mbar_try_wait_cluster(&bars->peer_done[prod], 0, 1000);
                    if (got) ip = static_cast<int>(bars->peer_issued[prod]);
                    else note_abort(bars, err, 12, peer_flag);
                    if (prod == 0 && q_loads > 0 &&
                        !mbar_wait(&bars->q_full, static_cast<uint32_t>(q_loads - 1) & 1u, kWaitIters))
                        note_abort(bars, err, 9, peer_flag);
                    const int hi = max(mine_end, ip);
                    for (int n = drain_from(hi); n < hi; ++n) {
                        if ((n & 1) != prod) continue;
                        uint64_t *fb = &bars->full[n % ST];
                        if (n < mine_end && n >= ip) mbar_complete_tx(fb, SLOT);         // the peer's part never comes
                        if (n >= mine_end && n < ip) mbar_arrive_expect_tx(fb, SLOT);    // only the peer's part
                        if (!mbar_wait(fb, static_cast<uint32_t>(n / ST) & 1u, kWaitIters))
                            note_abort(bars, err, 9, peer_flag);
                    }
                }
            } else {
                if (prod == 0 && q_loads > 0 &&
                    !mbar_wait(&bars->q_full, static_cast<uint32_t>(q_loads - 1) & 1u, kWaitIters))
                    note_abort(bars, err, 9, 0u);
                for (int n = drain_from(mine_end); n < mine_end; ++n)
                    if (mine(n) &&
                        !mbar_wait(&bars->full[n % ST], static_cast<uint32_t>(n / ST) & 1u, kWaitIters))
                        note_abort(bars, err, 9, 0u);
            }
            for (int n = drain_from(mine_end); n < mine_end; ++n)
                if (mine(n) &&
                    !mbar_wait(&bars->empty[n % ST], static_cast<uint32_t>(n / ST) & 1u, kWaitIters))
                    note_abort(bars, err, 9, PAIR ? peer_flag : 0u);
        }
    } else if (warp == 1 || warp == kPvWarp) {
        // ----------------------------------------------------------- MMA issue
        // Two issuing threads (of the leader, for a pair): warp 1 issues the
        // QK^T MMAs, warp kPvWarp the PV MMAs, so each one's waits and commits
        // overlap the other's MMAs on the tensor pipe.  Ring positions follow
        // the producers' order K_0, K_1, V_0, K_2, V_1, ..., V_T-1.  Warp 1 of
        // every CTA owns the TMEM allocation.
        const bool is_qk = warp == 1;
        if (lane == 0 && T > 0 && leader) {
            const uint32_t q_addr = smem_u32(sQ), ring_addr = smem_u32(sRing);
            // ring positions of tile t of a segment of Ts tiles (relative to
            // the segment's first position; a segment takes Ts (NSK + NSV))
            auto pos_k = [&](int t) { return t == 0 ? 0 : NSK + (t - 1) * (NSK + NSV); };
            auto pos_v = [&](int t, int Ts) {
                return t < Ts - 1 ? 2 * NSK + t * (NSK + NSV) : NSK + (Ts - 1) * (NSK + NSV);
            };
            // a slot is free once its MMAs are done (in both CTAs of a pair)
            auto release = [&](int slot) {
                if constexpr (PAIR) {
                    mma_commit_pair(smem_u32(&bars->empty[slot]));
                    mma_commit_pair(at_peer(&bars->empty[slot]));
                } else {
                    mma_commit(&bars->empty[slot]);
                }
            };
            auto commit_own = [&](uint64_t *bar) {
                if constexpr (PAIR) mma_commit_pair(smem_u32(bar));
                else mma_commit(bar);
            };
            auto commit_both = [&](uint64_t *bar) {
                commit_own(bar);
                if constexpr (PAIR) mma_commit_pair(at_peer(bar));
            };
            const uint32_t pf = PAIR ? peer_flag : 0u;
            bool ok = true;
            if (is_qk) {
                // S_t = Q K_t^T into TMEM buffer t % 2, over P_t-2: issued once
                // PV_t-2 has completed (s_free), the softmax of tile t-2 having
                // finished with S_t-2 before PV_t-2 was issued.
                constexpr uint32_t id_qk = idesc_f16(PAIR ? 256 : 128, 128, BF16 ? 1 : 0, 0, 0);
                int tg = 0, pbase = 0, qn = 0;
                for (int sgi = 0; sgi < nseg && ok; ++sgi) {
                const int Ts = sg_T[sgi];
                if (Ts == 0) continue;
                ok = wait_or_abort(bars, &bars->q_full, static_cast<uint32_t>(qn++) & 1u, err, 2, pf);
                for (int tl = 0; tl < Ts && ok; ++tl) {
                    const int t = tg + tl;                  // tile of the whole sequence
                    const int sb = t & 1;
                    if (t >= 2) ok = wait_or_abort(bars, &bars->s_free[sb], static_cast<uint32_t>((t - 2) >> 1) & 1u,
                                                   err, 3, pf, kPipeHintNs);
                    if (!ok) break;
                    tc_fence_after();
                    const int p0 = pbase + pos_k(tl);
                    for (int s = 0; s < NSK && ok; ++s) {
                        const int pos = p0 + s, slot = pos % ST;
                        ok = wait_or_abort(bars, &bars->full[slot], static_cast<uint32_t>(pos / ST) & 1u, err, 4, pf, kPipeHintNs);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t kb = ring_addr + slot * SLOT;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = sw128_desc(q_addr + s * kSlab + kk * 32, 16, 1024);
                            const uint64_t bd = sw128_desc(kb + kk * 32, 16, 1024);
                            if constexpr (PAIR) mma_f16_ss_pair(tm_s[sb], ad, bd, id_qk, (s | kk) != 0);
                            else mma_f16_ss(tm_s[sb], ad, bd, id_qk, (s | kk) != 0);
                        }
                        release(slot);
                    }
                    if (ok) commit_both(&bars->s_full[sb]);
                }
                tg += Ts;
                pbase += Ts * (NSK + NSV);
                }
            } else {
                int tg = 0, pbase = 0;
                for (int sgi = 0; sgi < nseg && ok; ++sgi) {
                const int Ts = sg_T[sgi];
                for (int tl = 0; tl < Ts && ok; ++tl) {
                    const int t = tg + tl;                  // tile of the whole sequence
                    ok = PAIR ? wait_or_abort_cluster(bars, &bars->p_full, static_cast<uint32_t>(t) & 1u, err, 5, pf,
                                                      kPipeHintNs)
                              : wait_or_abort(bars, &bars->p_full, static_cast<uint32_t>(t) & 1u, err, 5, pf, kPipeHintNs);
                    if (!ok) break;
                    tc_fence_after();
                    // V slots in runs of consecutive ring slots, one PV
                    // instruction per run and K step (single CTA: N = 64 x run
                    // length; pair: the tile's whole V group, N = DV over both
                    // CTAs).  P_t sits in TMEM over S_t: keys 64h + [0, 64) of
                    // the tile as P_hi in columns 64h + [0, 32) and P_lo in
                    // 64h + [32, 64), two 16-bit keys per column; each K step
                    // takes both terms.
                    int used = pbase + pos_v(tl, Ts);
                    for (int s = 0; s < NSV && ok;) {
                        const int slot0 = used % ST;
                        int len = 1;
                        while (s + len < NSV && slot0 + len < ST) ++len;
                        if (PAIR && len != NSV) {   // by construction a pair's V group never wraps
                            note_abort(bars, err, 13, pf);
                            ok = false;
                            break;
                        }
                        for (int j = 0; j < len && ok; ++j)
                            ok = wait_or_abort(bars, &bars->full[slot0 + j],
                                               static_cast<uint32_t>((used + j) / ST) & 1u, err, 6, pf, kPipeHintNs);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t vb = ring_addr + slot0 * SLOT;
                        if constexpr (PAIR) {
                            // this CTA's half of the columns: sub-slab j (16 KB)
                            // in slots 2j, 2j + 1; K step kk at kk * 2048 bytes
                            const uint32_t id_pv = idesc_f16(256, DV, BF16 ? 1 : 0, 0, 1);
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint32_t pa = tm_s[t & 1] + 64 * (kk >> 2) + 8 * (kk & 3);
                                const uint64_t bd = sw128_desc(vb + kk * 2048, kSlab, 1024);
                                mma_f16_ts_pair(tm_o, pa, bd, id_pv, (tl | kk) != 0);
                                mma_f16_ts_pair(tm_o, pa + 32, bd, id_pv, 1u);
                            }
                        } else {
                            const uint32_t id_pv = idesc_f16(128, 64 * len, BF16 ? 1 : 0, 0, 1);
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint32_t pa = tm_s[t & 1] + 64 * (kk >> 2) + 8 * (kk & 3);
                                const uint64_t bd = sw128_desc(vb + kk * 2048, kSlab, 1024);
                                mma_f16_ts(tm_o + s * 64, pa, bd, id_pv, (tl | kk) != 0);
                                mma_f16_ts(tm_o + s * 64, pa + 32, bd, id_pv, 1u);
                            }
                        }
                        for (int j = 0; j < len; ++j) release(slot0 + j);
                        used += len;
                        s += len;
                    }
                    if (!ok) break;
                    commit_both(&bars->o_done[t & 1]);
                    commit_own(&bars->s_free[t & 1]);   // S_t / P_t buffer free once PV_t is done
                }
                tg += Ts;
                pbase += Ts * (NSK + NSV);
                }
            }
            // Drain: all MMAs issued by this thread have completed.
            uint64_t *dr = is_qk ? &bars->drain : &bars->drain_pv;
            commit_own(dr);
            if (!mbar_wait(dr, 0, kWaitIters)) note_abort(bars, err, 10, pf);
        }
    } else if (warp >= 2) {
        // ---------------------------------------------- softmax and epilogue
        // Eight warps: warp w reads TMEM lanes 32*(w%4).. (its 32 rows) and owns
        // one 64-key half of each tile (chunks 2*half, 2*half+1) and one half of
        // the O columns; the two warps of a quarter combine row maxima and sums
        // through shared memory with a 64-thread named barrier.
        const int sw = warp - 2;
        const int half = sw >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;              // row within the tile
        int rg = 0, qi = 0;                             // row within the KV group, query (tree node)
        const float *mrow = nullptr;                    // its mask row
        auto rows_of_segment = [&]() {
            rg = rt * RT + r;
            qi = rg % a.L;
            mrow = (IMPLICIT || a.mask == nullptr) ? nullptr : a.mask + static_cast<size_t>(qi) * a.stride;
        };
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const int last0 = a.N - a.L;
        constexpr int DVH = DV / 2;                     // O columns of this warp
        auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(1 + quarter) : "memory"); };

        ChunkWalk walk;
        float m_run = -INFINITY, l_half = 0.0f;         // running max (log2 units), this half's sum
        bool ok = true;
        const float scale2 = a.scale * kLog2e;
        // A wait's outcome is made warp-uniform (TMEM loads/stores are warp-
        // collective), and the named barriers run in every iteration even after
        // a failed wait, so no softmax warp can be left at a barrier.
        auto wait_all = [&](uint64_t *bar, uint32_t parity, int code) -> bool {
            const bool w = ok && wait_or_abort(bars, bar, parity, err, code, PAIR ? peer_flag : 0u);
            return __all_sync(0xffffffffu, w);
        };
        int tg = 0;                                     // tiles of earlier segments
        for (int sgi = 0; sgi < nseg; ++sgi) {
        const int Ts = sg_T[sgi];
        enter_segment(sgi);
        rows_of_segment();
        walk.init(a.cls, sg_cb[sgi], sg_ce[sgi]);
        m_run = -INFINITY;
        l_half = 0.0f;
        for (int tl = 0; tl < Ts; ++tl) {
            const int t = tg + tl;                      // tile of the whole sequence
            int chunk[4], ccls[4];
            for (int c = 0; c < 4; ++c) chunk[c] = walk.next(&ccls[c]);
            const int ch0 = half ? chunk[2] : chunk[0], ch1 = half ? chunk[3] : chunk[1];
            const int cl0 = half ? ccls[2] : ccls[0], cl1 = half ? ccls[3] : ccls[1];
            // mask of this half's first mixed chunk, fetched before waiting for S
            int mixed = -1;
            float mpre[32];
            if (!IMPLICIT) {
                mixed = (ch0 >= 0 && cl0 == kChunkMixed) ? 0 : ((ch1 >= 0 && cl1 == kChunkMixed) ? 1 : -1);
                if (mixed >= 0) explicit_chunk(a, mrow, qi, (mixed ? ch1 : ch0) * 32, mpre);
            }
            const int sb = t & 1;
            ok = wait_all(&bars->s_full[sb], (static_cast<uint32_t>(t) >> 1) & 1u, 7);
            tc_fence_after();

            // pass 1: logits (log2 units) of this half's two chunks, written back
            // over S in TMEM, and their row maximum
            float pmax = -INFINITY;
#pragma unroll 1
            for (int cc = 0; cc < (ok ? 2 : 0); ++cc) {
                const int ch = cc ? ch1 : ch0, ccl = cc ? cl1 : cl0;
                const uint32_t col = tm_s[sb] + lane_off + (2 * half + cc) * 32;
                uint32_t v[32];
                tmem_ld32(col, v);
                tmem_wait_ld();
                const int key0 = ch * 32;
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                if (ch >= 0 && ccl == kChunkAllAttended && key0 + 32 <= a.N) {
                    // every cell attended: mask 0, logit = qk * scale
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float lg = __uint_as_float(v[e]) * scale2;
                        m4[e & 3] = fmaxf(m4[e & 3], lg);
                        v[e] = __float_as_uint(lg);
                    }
                } else if (ch < 0) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(-INFINITY);
                } else {
                    float mv[32];
                    if (IMPLICIT) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int key = key0 + e;
                            mv[e] = (key < a.N && key >= a.window_start && key <= last0 + qi) ? 0.0f : kMasked;
                        }
                    } else if (ccl == kChunkAllAttended) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) mv[e] = key0 + e < a.N ? 0.0f : kMasked;
                    } else if (cc == mixed) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) mv[e] = mpre[e];
                    } else {
                        explicit_chunk(a, mrow, qi, key0, mv);
                    }
                    bool live = false;
#pragma unroll
                    for (int e = 0; e < 32; ++e) live |= mv[e] > kMasked;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        // logit = fma(qk, scale, mask) (the pages' form), in log2 units
                        const float lg = live ? fmaf(__uint_as_float(v[e]), a.scale, mv[e]) * kLog2e : -INFINITY;
                        m4[e & 3] = fmaxf(m4[e & 3], lg);
                        v[e] = __float_as_uint(lg);
                    }
                }
                pmax = fmaxf(pmax, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])));
                tmem_st32(col, v);
            }
            tmem_wait_st();
            bars->xrow[t & 1][half][r] = pmax;
            pair_sync();
            const float rmax = fmaxf(pmax, bars->xrow[t & 1][half ^ 1][r]);

            // online softmax with lazy rescaling (same decision in both halves)
            float alpha = 1.0f;
            if (rmax > m_run + kRescaleSlack2) {
                alpha = fast_exp2(m_run - rmax);        // 0 when m_run = -inf
                l_half *= alpha;
                m_run = rmax;
            }
            const float m_use = m_run == -INFINITY ? 0.0f : m_run;   // dead row: all logits -inf, P = 0

            // A rescale needs O stable: wait for PV of the previous tile (only
            // then; P_t has a TMEM buffer of its own).  Waiting for tile t-1 on
            // o_done[(t-1) % 2] is unambiguous: S_t was issued after PV_t-2 was
            // done, so that barrier's phase is the one of tile t-1.
            if (tl > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
                ok = wait_all(&bars->o_done[(t - 1) & 1], (static_cast<uint32_t>(t - 1) >> 1) & 1u, 8);
                tc_fence_after();
                if (ok) {
#pragma unroll 1
                    for (int c = 0; c < DVH / 32; ++c) {
                        uint32_t rr[32];
                        const uint32_t col = tm_o + lane_off + half * DVH + c * 32;
                        tmem_ld32(col, rr);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
                        tmem_st32(col, rr);
                    }
                    tmem_wait_st();
                }
            }
            // pass 2: P = 2^(logit - M) as two 16-bit terms of the K/V type,
            // P_hi = rn(P) and P_lo = rn(P - P_hi), written back into TMEM over
            // this half's logits (P_hi in columns 64 * half + [0, 32), P_lo in
            // 64 * half + [32, 64); two keys per column, the lower key in the
            // low 16 bits), where PV reads them as A operands.  The row sum adds
            // P in f32 (P_hi + P_lo equals it to 2^-16 relative).
            float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            uint32_t pw[32], pl[32];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t v[32];
                if (ok) {
                    tmem_ld32(tm_s[sb] + lane_off + (2 * half + cc) * 32, v);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(-INFINITY);
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float p0 = fast_exp2(__uint_as_float(v[2 * j]) - m_use);
                    const float p1 = fast_exp2(__uint_as_float(v[2 * j + 1]) - m_use);
                    const uint32_t w = pack2(p0, p1, BF16);
                    pw[cc * 16 + j] = w;
                    pl[cc * 16 + j] = pack2(p0 - lo16(w, BF16), p1 - hi16(w, BF16), BF16);
                    ps[(2 * j) & 7] += p0;
                    ps[(2 * j + 1) & 7] += p1;
                }
            }
            if (ok) {
                tmem_st32(tm_s[sb] + lane_off + 64 * half, pw);
                tmem_st32(tm_s[sb] + lane_off + 64 * half + 32, pl);
                tmem_wait_st();
            }
            l_half += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
            tc_fence_before();
            __syncwarp();
            if (lane == 0 && ok) {
                if (PAIR && !leader) mbar_arrive_remote(at_leader(&bars->p_full));
                else mbar_arrive(&bars->p_full);
            }
        }
        if (flat) {
            // ---- end of a flattened segment: its partial (unnormalized O of
            // this CTA's rows and O half, and (S, M)) goes from TMEM straight
            // to its slot.  The next segment's first PV starts O over only
            // after these warps signal P of that tile, i.e. after these loads.
            const int tlast = tg + Ts - 1;
            if (Ts > 0) {
                ok = wait_all(&bars->o_done[tlast & 1], (static_cast<uint32_t>(tlast) >> 1) & 1u, 8);
                tc_fence_after();
            }
            const int px = (tg + Ts) & 1;               // the exchange buffer of the next tile
            bars->xrow[px][half][r] = l_half;
            pair_sync();
            const float l_run = l_half + bars->xrow[px][half ^ 1][r];
            pair_sync();                                // both read it before the next tile writes it
            const int nrows = a.H * a.L;
            const size_t rid2 = static_cast<size_t>(qi) * a.H + kh * a.g + rg / a.L;
            const bool row_ok = r < rows_here;
            const size_t slot = static_cast<size_t>(sg_slot[sgi]);
            if (Ts > 0 && ok) {
#pragma unroll 1
                for (int c = 0; c < DVH / 32; ++c) {
                    uint32_t rr[32];
                    tmem_ld32(tm_o + lane_off + half * DVH + c * 32, rr);
                    tmem_wait_ld();
                    if (row_ok) {
                        float4 *dst = reinterpret_cast<float4 *>(a.part_o + (slot * nrows + rid2) * D + os * DV +
                                                                 half * DVH + c * 32);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            dst[e] = make_float4(__uint_as_float(rr[4 * e]), __uint_as_float(rr[4 * e + 1]),
                                                 __uint_as_float(rr[4 * e + 2]), __uint_as_float(rr[4 * e + 3]));
                    }
                }
            }
            if (os == 0 && half == 0 && row_ok) {
                float2 *ml = reinterpret_cast<float2 *>(a.part_ml);
                ml[slot * nrows + rid2] =
                    make_float2(Ts > 0 ? l_run : 0.0f, m_run == -INFINITY ? kMInit : m_run * kLn2);
                // the unit's slots no group fills hold no keys (S = 0: the merge skips them)
                if (sg_last[sgi])
                    for (int s2 = sg_used[sgi]; s2 < a.nwg; ++s2)
                        ml[static_cast<size_t>(s2) * nrows + rid2] = make_float2(0.0f, kMInit);
            }
        }
        tg += Ts;
        }
        if (flat) {
            pdl_launch_dependents();
        } else {
        if (T > 0) {
            ok = wait_all(&bars->o_done[(T - 1) & 1], (static_cast<uint32_t>(T - 1) >> 1) & 1u, 8);
            tc_fence_after();
        }
        // epilogue: row sum of both halves; the unnormalized O rows and the
        // row's (S, M) are staged in shared memory (free once the last MMA is
        // done; O rows padded by 16 bytes) for the store / merge phase below
        pdl_launch_dependents();
        bars->xrow[T & 1][half][r] = l_half;
        pair_sync();
        const float l_run = l_half + bars->xrow[T & 1][half ^ 1][r];
        const bool have_o = ok && T > 0;
        // a final row stored straight from the stage (no merge in the cluster)
        // is normalized here
        const float row_sc = (cx == 1 && a.n_part == 0) ? (l_run == 0.0f ? 0.0f : 1.0f / l_run) : 1.0f;
        float *stage = reinterpret_cast<float *>(sm);
#pragma unroll 1
        for (int c = 0; c < DVH / 32; ++c) {
            uint32_t rr[32];
            if (have_o) {
                tmem_ld32(tm_o + lane_off + half * DVH + c * 32, rr);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) rr[e] = 0u;
            }
            float *srow = stage + r * SROW + half * DVH + c * 32;
#pragma unroll
            for (int e = 0; e < 32; e += 4)
                *reinterpret_cast<float4 *>(srow + e) =
                    make_float4(__uint_as_float(rr[e]) * row_sc, __uint_as_float(rr[e + 1]) * row_sc,
                                __uint_as_float(rr[e + 2]) * row_sc, __uint_as_float(rr[e + 3]) * row_sc);
        }
        if (half == 0)
            reinterpret_cast<float2 *>(stage + 128 * SROW)[r] =
                make_float2(l_run, m_run == -INFINITY ? kMInit : m_run * kLn2);   // (S, M), natural log
        fence_proxy_async_smem();   // the staged rows may leave by bulk copy
        }
    }

    // ------------------------------------------------------ store or merge
    // With an x extent, after the cluster barrier every CTA's staged rows are
    // visible to its peers.  Without one each CTA stores its own rows; otherwise CTA
    // x of the cluster takes rows [x * n, (x + 1) * n) of the tile and merges
    // them over the cx splits of the cluster (log-sum-exp weights, loads from
    // the peers' shared memory).  With n_part == 0 the merged rows are final
    // (normalized output); else they are partial slot split / cx.
    tc_fence_before();
    __syncthreads();
    if (cx > 1) cluster_sync();   // the merge reads the peers' staged rows (cx is uniform in a cluster)
    const bool epi_warp = warp >= 2 && warp < kProd1Warp;   // the softmax warps
    if (epi_warp && cx == 1 && !flat) {
        // No merge in the cluster: each staged row (final and normalized, or
        // partial slot `split` with its (S, M)) leaves by one bulk copy issued
        // by its own thread; a destination off a 16-byte boundary is written
        // with plain stores instead.
        constexpr int F4 = DV / 4;                      // float4 per row
        const int t2 = tid - 64;
        const int nrows = a.H * a.L;
        const bool final_out = a.n_part == 0;
        const float *stage = reinterpret_cast<const float *>(sm);
        const float2 *stage_ml = reinterpret_cast<const float2 *>(stage + 128 * SROW);
        bool issued = false;
        for (int rr = t2; rr < rows_here; rr += 256) {
            const int rg2 = rt * RT + rr;
            const size_t rid2 = static_cast<size_t>(rg2 % a.L) * a.H + kh * a.g + rg2 / a.L;
            float *dst = final_out ? a.out + rid2 * D + os * DV
                                   : a.part_o + (static_cast<size_t>(split) * nrows + rid2) * D + os * DV;
            const float *src = stage + rr * SROW;
            if ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
                bulk_store(dst, src, DV * 4);
                issued = true;
            } else {
                for (int c4 = 0; c4 < F4; ++c4) {
                    const float4 o = *reinterpret_cast<const float4 *>(src + 4 * c4);
                    dst[4 * c4] = o.x; dst[4 * c4 + 1] = o.y; dst[4 * c4 + 2] = o.z; dst[4 * c4 + 3] = o.w;
                }
            }
        }
        if (issued) {
            bulk_commit();
            bulk_wait_all();   // the stage is read and the rows written before the CTA moves on
        }
        if (!final_out && os == 0)
            for (int rr = t2; rr < rows_here; rr += 256) {
                const int rg2 = rt * RT + rr;
                const size_t rid2 = static_cast<size_t>(rg2 % a.L) * a.H + kh * a.g + rg2 / a.L;
                reinterpret_cast<float2 *>(a.part_ml)[static_cast<size_t>(split) * nrows + rid2] = stage_ml[rr];
            }
    } else if (epi_warp && !flat) {
        const int sw = warp - 2;
        const int nrows = a.H * a.L;
        const bool final_out = a.n_part == 0;
        const float *stage = reinterpret_cast<const float *>(sm);
        const uint32_t stage_sa = smem_u32(stage);
        const uint32_t ml_sa = stage_sa + 128 * SROW * 4;
        const int slot = split / cx;
        const int rows_per = (rows_here + cx - 1) / cx;
        const int r0 = cxi * rows_per, r1 = min(rows_here, r0 + rows_per);
        constexpr int C4 = DV / 128;                    // float4 columns per lane
        for (int rr = r0 + sw; rr < r1; rr += 8) {
            const int rg2 = rt * RT + rr;
            const size_t rid2 = static_cast<size_t>(rg2 % a.L) * a.H + kh * a.g + rg2 / a.L;
            // up to 16 splits: lane p < cx holds split p's (S, M); the weighted
            // rows are summed in rounds of 8, each round's remote loads all
            // issued before any is used
            float2 ml = make_float2(0.0f, -FLT_MAX);
            if (lane < cx) ml = ld_dsmem_f2(mapa_shared(ml_sa + rr * 8, lane));
            const float mstar = warp_max(lane < cx ? ml.y : -FLT_MAX);
            const float wp = lane < cx ? expf(ml.y - mstar) : 0.0f;
            const float sstar = warp_sum(lane < cx ? ml.x * wp : 0.0f);
            const float inv = (sstar == 0.0f) ? 0.0f : 1.0f / sstar;
            float4 acc[C4];
#pragma unroll
            for (int j = 0; j < C4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
            for (int p0 = 0; p0 < cx; p0 += 8) {
                float4 v[8][C4];
#pragma unroll
                for (int p = 0; p < 8; ++p) {
                    if (p0 + p >= cx) break;
#pragma unroll
                    for (int j = 0; j < C4; ++j) {
                        const uint32_t off = stage_sa + (rr * SROW + 4 * (lane + 32 * j)) * 4;
                        v[p][j] = cx > 1 ? ld_dsmem_f4(mapa_shared(off, p0 + p))
                                         : *reinterpret_cast<const float4 *>(stage + rr * SROW + 4 * (lane + 32 * j));
                    }
                }
#pragma unroll
                for (int p = 0; p < 8; ++p) {
                    if (p0 + p >= cx) break;
                    const float w = __shfl_sync(0xffffffffu, wp, p0 + p);
#pragma unroll
                    for (int j = 0; j < C4; ++j) {
                        acc[j].x += w * v[p][j].x; acc[j].y += w * v[p][j].y;
                        acc[j].z += w * v[p][j].z; acc[j].w += w * v[p][j].w;
                    }
                }
            }
            float *dst = final_out ? a.out + rid2 * D + os * DV
                                   : a.part_o + (static_cast<size_t>(slot) * nrows + rid2) * D + os * DV;
#pragma unroll
            for (int j = 0; j < C4; ++j) {
                float4 o = acc[j];
                if (final_out) { o.x *= inv; o.y *= inv; o.z *= inv; o.w *= inv; }
                *reinterpret_cast<float4 *>(dst + 4 * (lane + 32 * j)) = o;
            }
            if (!final_out && lane == 0 && os == 0) {
                a.part_ml[(static_cast<size_t>(slot) * nrows + rid2) * 2 + 0] = sstar;
                a.part_ml[(static_cast<size_t>(slot) * nrows + rid2) * 2 + 1] = mstar;
            }
        }
    }

    __syncthreads();
    tc_fence_before();
    cluster_sync();                                     // peers are done with this CTA's shared memory and TMEM
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if constexpr (PAIR) tmem_dealloc_pair(tmem, 512);
        else tmem_dealloc(tmem, 512);
    }
}

// Clusters above 8 CTAs need the kernel's non-portable cluster size allowed.
template <typename Kern>
cudaError_t allow_big_clusters_once(Kern kern, unsigned long long *done_mask) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) __atomic_fetch_or(done_mask, bit, __ATOMIC_ACQ_REL);
    return e;
}

// Clusters of `size` (<= 16) CTAs of this kernel that the current device can
// hold at once (the kernel is shared-memory bound to one CTA per SM, equally
// for all instantiations); cached per device.
static int max_active_clusters(int size) {
    static int cache[64][17];
    int dev = 0;
    if (size < 1 || size > 16) return 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) { cudaGetLastError(); return 0; }
    const int idx = size;
    int n = __atomic_load_n(&cache[dev][idx], __ATOMIC_ACQUIRE);
    if (n > 0) return n;
    auto kern = tree_tc_kernel<256, false, false, false>;
    static unsigned long long done = 0;
    if (set_smem_limit_once(kern, TcCfg<256, false>::SMEM, &done) != cudaSuccess) { cudaGetLastError(); return 0; }
    static unsigned long long big = 0;
    if (size > 8 && allow_big_clusters_once(kern, &big) != cudaSuccess) { cudaGetLastError(); return 0; }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(size, 1, 1);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = TcCfg<256, false>::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = size;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) { cudaGetLastError(); n = 0; }
    if (n > 0) __atomic_store_n(&cache[dev][idx], n, __ATOMIC_RELEASE);
    return n;
}

}  // namespace

// Splits merged inside one cluster.  The CTA-pair form's cluster is the pair:
// no in-cluster merge (1).
// Otherwise all splits of a (row tile, O half, KV head) along x when they fit
// in one cluster (at most 8 CTAs) and every cluster of the grid fits on the
// device at once, so the merge completes inside the cluster and no partials
// are written (a partial in-cluster merge costs more in remote loads than it
// saves in partial traffic); else clusters of one.  cy is always 1.
void tree_tc_cluster_shape(const TreeArgs &a, int *cx, int *cy) {
    *cx = 1;
    *cy = 1;
    if (tree_tc_pairs(a.R, a.D)) return;
    // every cluster resident at once: clusters = row tiles x O halves x KV heads
    const long clusters = static_cast<long>(tree_tc_row_ctas(a.R, a.D)) * (a.D == 512 ? 2 : 1) * a.Hk;
    if (a.nwg > 1 && a.nwg <= 16) {
        const int n = max_active_clusters(a.nwg);
        if (n > 0 && clusters <= n) *cx = a.nwg;
    }
}

namespace {

template <int D, bool BF16, bool IMPLICIT, bool PAIR>
cudaError_t launch_tc_one(const TreeArgs &a, const TcMaps &maps, cudaStream_t s) {
    using Cfg = TcCfg<D, PAIR>;
    auto kern = tree_tc_kernel<D, BF16, IMPLICIT, PAIR>;
    static unsigned long long done = 0, big = 0;
    cudaError_t e = set_smem_limit_once(kern, Cfg::SMEM, &done);
    if (e == cudaSuccess && a.cluster_x > 8) e = allow_big_clusters_once(kern, &big);
    if (e != cudaSuccess) return e;
    constexpr unsigned halves = D / Cfg::DV;
    const unsigned n_ct = static_cast<unsigned>(tree_tc_row_ctas(a.R, D));
    dim3 grid;
    unsigned cx, cy = 1;
    if (PAIR) {
        grid = a.flat_groups > 0 ? dim3(2, static_cast<unsigned>(a.flat_groups) * halves, 1)
                                 : dim3(n_ct, static_cast<unsigned>(a.nwg) * halves, a.Hk);
        cx = 2;
    } else {
        int mx, my;
        tree_tc_cluster_shape(a, &mx, &my);
        grid = dim3(a.nwg, n_ct * halves, a.Hk);
        cx = static_cast<unsigned>(mx);
    }
    e = launch_pdl_cluster(kern, grid, dim3(kTcThreads), Cfg::SMEM, s, cx, cy, a, maps);
    count_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int D, bool BF16, bool IMPLICIT>
cudaError_t launch_tc_rows(const TreeArgs &a, const TcMaps &maps, cudaStream_t s) {
    if constexpr (D == 512) {
        if (tree_tc_pairs(a.R, D)) return launch_tc_one<D, BF16, IMPLICIT, true>(a, maps, s);
    }
    return launch_tc_one<D, BF16, IMPLICIT, false>(a, maps, s);
}

template <bool BF16>
cudaError_t launch_tc_typed(const TreeArgs &a, const TcMaps &maps, cudaStream_t s) {
    const bool imp = a.mask == nullptr && a.anc == nullptr;
    switch (a.D) {
        case 128: return imp ? launch_tc_rows<128, BF16, true>(a, maps, s) : launch_tc_rows<128, BF16, false>(a, maps, s);
        case 256: return imp ? launch_tc_rows<256, BF16, true>(a, maps, s) : launch_tc_rows<256, BF16, false>(a, maps, s);
        case 512: return imp ? launch_tc_rows<512, BF16, true>(a, maps, s) : launch_tc_rows<512, BF16, false>(a, maps, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_tree_tc(const TreeArgs &a, const TcMaps &maps, int kv_type, cudaStream_t s) {
    if (kv_type == kKvF16) return launch_tc_typed<false>(a, maps, s);
    if (kv_type == kKvBF16) return launch_tc_typed<true>(a, maps, s);
    return cudaErrorInvalidValue;
}

}  // namespace ta
