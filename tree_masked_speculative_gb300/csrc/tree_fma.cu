// CUDA-core tree-verify attention main pass.
//
// Semantics follow mlx-native tree_attention.metal (tree_attention_impl):
// 32-key chunks, a chunk skipped for a row when all its mask cells are
// <= -65504, logit = fma(qk, scale, mask), online softmax per chunk
// (M' = max(M, max_j s_j), S = S * e^(M - M') + sum_j e^(s_j - M'),
// O = O * e^(M - M') + sum_j e^(s_j - M') V_j), and per-split partials
// (O, S, M) merged by the reduce pass.
//
// GB300 layout (not the pages' one-row-per-threadgroup mapping): one CTA per
// (KV head, group of up to 16 query rows of that head, split).  Each live
// chunk's K and V rows are loaded from HBM once into shared memory and used
// by every row of the group; the split partitions the list of live chunks
// (chunks that at least one row attends, from the compaction pass), so dead
// chunks are never loaded.  This kernel is the path for f32 KV caches and for
// KV heads serving fewer than 16 query rows; f16/bf16 caches with >= 16 rows
// per KV head run on the tensor-core kernel.
#include "ta_internal.cuh"

namespace ta {

namespace {

constexpr int kThreads = 128;
constexpr int kRB = kFmaRowsPerCta;   // rows per CTA, 4 per warp

template <int D>
struct FmaSmem {
    static constexpr int kQ = kRB * D;          // sQ [16][D]
    static constexpr int kK = 32 * (D + 1);     // sK [32][D+1] (padded: lane = key)
    static constexpr int kV = 32 * D;           // sV [32][D]
    static constexpr size_t bytes = sizeof(float) * (kQ + kK + kV) + sizeof(int) * (2 * 128 + 16);
};

// Block-wide exclusive scan of a 0/1 flag over 128 threads; returns the
// exclusive prefix and writes the total to *total.
__device__ __forceinline__ int block_scan128(int flag, int *s_warp, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned b = __ballot_sync(0xffffffffu, flag);
    int excl = __popc(b & ((1u << lane) - 1u));
    if (lane == 0) s_warp[warp] = __popc(b);
    __syncthreads();
    int base = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        int c = s_warp[w];
        if (w < warp) base += c;
        tot += c;
    }
    __syncthreads();
    *total = tot;
    return base + excl;
}

template <int D, typename KV_T, bool IMPLICIT>
__global__ void __launch_bounds__(kThreads) tree_fma_kernel(const TreeArgs a) {
    constexpr int DPL = D / 32;                 // output dims per lane
    constexpr int EPV = Vec16<KV_T>::N;         // KV elements per 16-byte vector
    constexpr int VPR = D / EPV;                // vectors per KV row
    extern __shared__ __align__(16) float smem[];
    float *sQ = smem;
    float *sK = sQ + FmaSmem<D>::kQ;
    float *sV = sK + FmaSmem<D>::kK;
    int *sList = reinterpret_cast<int *>(sV + FmaSmem<D>::kV);
    int *sCls = sList + 128;
    int *sWarp = sCls + 128;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, r0 = blockIdx.y * kRB, kh = blockIdx.z;
    pdl_wait();                                 // chunk classes are ready

    // Q rows of this group: global row kh * R + r0 + rr, r = j * L + i.
    for (int idx = tid; idx < kRB * (D / 4); idx += kThreads) {
        const int rr = idx / (D / 4), c4 = idx % (D / 4);
        float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r0 + rr < a.R)
            val = __ldg(reinterpret_cast<const float4 *>(a.q + ((size_t)kh * a.R + r0 + rr) * D) + c4);
        reinterpret_cast<float4 *>(sQ)[idx] = val;
    }

    int row_i[4], row_h[4];
    bool row_ok[4];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
        const int r = r0 + warp * 4 + rr;
        row_ok[rr] = r < a.R;
        const int j = row_ok[rr] ? r / a.L : 0;
        row_i[rr] = row_ok[rr] ? r % a.L : 0;
        row_h[rr] = kh * a.g + j;
    }
    float M[4], S[4], O[4][DPL];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
        M[rr] = kMInit;
        S[rr] = 0.0f;
#pragma unroll
        for (int t = 0; t < DPL; ++t) O[rr][t] = 0.0f;
    }

    // Live chunks (any row attends) and this split's share of them.
    int n_live = 0;
    for (int base = 0; base < a.n_chunks; base += kThreads) {
        const int c = base + tid;
        int tot;
        block_scan128(c < a.n_chunks && a.cls[c] != kChunkDead, sWarp, &tot);
        n_live += tot;
    }
    const int cps = (n_live + a.nwg - 1) / a.nwg;
    const int lo = split * cps, hi = min(n_live, lo + cps);

    const KV_T *kbase = reinterpret_cast<const KV_T *>(a.k) + (size_t)kh * a.C * D;
    const KV_T *vbase = reinterpret_cast<const KV_T *>(a.v) + (size_t)kh * a.C * D;
    const int last0 = a.N - a.L;   // implicit mask: row i attends keys <= last0 + i

    int rank_base = 0;
    for (int base = 0; base < a.n_chunks && rank_base < hi; base += kThreads) {
        const int c = base + tid;
        const int cl = c < a.n_chunks ? a.cls[c] : kChunkDead;
        int tot;
        const int excl = block_scan128(cl != kChunkDead, sWarp, &tot);
        const int rank = rank_base + excl;
        const int first = max(lo, rank_base);
        if (cl != kChunkDead && rank >= lo && rank < hi) {
            sList[rank - first] = c;
            sCls[rank - first] = cl;
        }
        const int n_mine = max(0, min(hi, rank_base + tot) - first);
        rank_base += tot;
        __syncthreads();

        for (int e = 0; e < n_mine; ++e) {
            const int chunk = sList[e];
            const int ccls = sCls[e];
            const int key0 = chunk * 32;
            // K and V rows key0..key0+31 -> shared f32 (zeros past kv_seq_len)
            for (int idx = tid; idx < 32 * VPR; idx += kThreads) {
                const int rk = idx / VPR, cv = idx % VPR;
                uint4 ku = make_uint4(0, 0, 0, 0), vu = make_uint4(0, 0, 0, 0);
                if (key0 + rk < a.N) {
                    ku = __ldg(reinterpret_cast<const uint4 *>(kbase + (size_t)(key0 + rk) * D) + cv);
                    vu = __ldg(reinterpret_cast<const uint4 *>(vbase + (size_t)(key0 + rk) * D) + cv);
                }
                float kf[EPV], vf[EPV];
                Vec16<KV_T>::expand(ku, kf);
                Vec16<KV_T>::expand(vu, vf);
#pragma unroll
                for (int x = 0; x < EPV; ++x) {
                    sK[rk * (D + 1) + cv * EPV + x] = kf[x];
                    sV[rk * D + cv * EPV + x] = vf[x];
                }
            }
            __syncthreads();

            // QK for the warp's 4 rows; lane = key of the chunk.
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            const float *krow = sK + lane * (D + 1);
            const float *q0 = sQ + (warp * 4) * D;
#pragma unroll 4
            for (int d = 0; d < D; ++d) {
                const float kv = krow[d];
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) acc[rr] = fmaf(q0[rr * D + d], kv, acc[rr]);
            }
            const int key = key0 + lane;
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                if (!row_ok[rr]) continue;
                float mv;
                if (key >= a.N) {
                    mv = kMasked;
                } else if (IMPLICIT) {
                    mv = (key >= a.window_start && key <= last0 + row_i[rr]) ? 0.0f : kMasked;
                } else {
                    mv = (ccls == kChunkAllAttended)
                             ? 0.0f
                             : explicit_cell(a, a.mask == nullptr ? nullptr : a.mask + (size_t)row_i[rr] * a.stride,
                                             row_i[rr], key);
                }
                if (!__any_sync(0xffffffffu, mv > kMasked)) continue;   // chunk dead for this row
                const float s = fmaf(acc[rr], a.scale, mv);
                const float m_old = M[rr];
                M[rr] = fmaxf(m_old, warp_max(s));
                const float ms = expf(m_old - M[rr]);
                const float vs = expf(s - M[rr]);
                S[rr] = S[rr] * ms + warp_sum(vs);
#pragma unroll
                for (int t = 0; t < DPL; ++t) O[rr][t] *= ms;
#pragma unroll 4
                for (int kk = 0; kk < 32; ++kk) {
                    const float wgt = __shfl_sync(0xffffffffu, vs, kk);
                    const float *vr = sV + kk * D + lane;
#pragma unroll
                    for (int t = 0; t < DPL; ++t) O[rr][t] = fmaf(wgt, vr[32 * t], O[rr][t]);
                }
            }
            __syncthreads();
        }
    }

    // Partials (or the normalized output when there is a single split).
    const int nrows = a.H * a.L;
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
        if (!row_ok[rr]) continue;
        const size_t rid = (size_t)row_i[rr] * a.H + row_h[rr];
        if (a.nwg == 1) {
            const float inv = (S[rr] == 0.0f) ? 0.0f : 1.0f / S[rr];
            float *dst = a.out + rid * D + lane;
#pragma unroll
            for (int t = 0; t < DPL; ++t) dst[32 * t] = O[rr][t] * inv;
        } else {
            float *dst = a.part_o + ((size_t)split * nrows + rid) * D + lane;
#pragma unroll
            for (int t = 0; t < DPL; ++t) dst[32 * t] = O[rr][t];
            if (lane == 0) {
                a.part_ml[((size_t)split * nrows + rid) * 2 + 0] = S[rr];
                a.part_ml[((size_t)split * nrows + rid) * 2 + 1] = M[rr];
            }
        }
    }
}

template <int D, typename KV_T, bool IMPLICIT>
cudaError_t launch_one(const TreeArgs &a, cudaStream_t s) {
    auto kern = tree_fma_kernel<D, KV_T, IMPLICIT>;
    const size_t smem = FmaSmem<D>::bytes;
    static unsigned long long done = 0;
    cudaError_t e = set_smem_limit_once(kern, smem, &done);
    if (e != cudaSuccess) return e;
    dim3 grid(a.nwg, (a.R + kRB - 1) / kRB, a.Hk);
    e = launch_pdl(kern, grid, dim3(kThreads), smem, s, a);
    count_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename KV_T>
cudaError_t launch_typed(const TreeArgs &a, cudaStream_t s) {
    const bool imp = a.mask == nullptr && a.anc == nullptr;
    switch (a.D) {
        case 128: return imp ? launch_one<128, KV_T, true>(a, s) : launch_one<128, KV_T, false>(a, s);
        case 256: return imp ? launch_one<256, KV_T, true>(a, s) : launch_one<256, KV_T, false>(a, s);
        case 512: return imp ? launch_one<512, KV_T, true>(a, s) : launch_one<512, KV_T, false>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_tree_fma(const TreeArgs &a, int kv_type, cudaStream_t s) {
    switch (kv_type) {
        case kKvF32: return launch_typed<float>(a, s);
        case kKvF16: return launch_typed<__half>(a, s);
        case kKvBF16: return launch_typed<__nv_bfloat16>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ta
