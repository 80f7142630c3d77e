// Mask compaction (per-32-key-chunk classification) and the split-merge pass
// of the tree-verify attention.
//
// Classification: mlx-native tree_attention.metal skips a 32-key chunk for a
// query row when every mask cell of the chunk is <= -65504 (main kernel, mask
// read and early exit).  Here the whole mask is classified once per call so
// that the main kernels never load K/V of a chunk that no row attends and never
// read mask cells of a chunk that every row fully attends.
//
// Merge: the pages reuse flash_attn_vec_reduce without showing it
// (tree_attention.rs, reduce pass); this is the log-sum-exp merge of the NWG
// (S, M, O) partials of each row.
#include "ta_internal.cuh"

namespace ta {

// Prep pass, one launch: blocks [0, n_chunks) classify one 32-key chunk each
// (dead if no (row, key < N) cell is attended (> -65504), all-attended if every
// (row, key < N) cell equals 0.0, else mixed; lane = key, the L rows spread
// over the 8 warps); the remaining blocks write the 16-bit copy of Q for the
// tensor-core kernel; block 0 clears the error word.
constexpr int kPrepThreads = 256;
constexpr int kQ16PerBlock = kPrepThreads * 8;

__global__ void __launch_bounds__(kPrepThreads) tree_prep_kernel(const TreeArgs a, int n_cls_blocks) {
    pdl_launch_dependents();
    if (blockIdx.x == 0 && threadIdx.x == 0 && a.err != nullptr) {
        a.err[0] = 0;          // error word
        a.err[1] = a.n_part;   // partial slots the main pass leaves for the merge
    }
    if (static_cast<int>(blockIdx.x) >= n_cls_blocks) {
        // Q [H*L, D] f32 -> 16-bit (round to nearest), 8 elements per thread
        const size_t total = static_cast<size_t>(a.H) * a.L * a.D;
        const size_t i8 = (static_cast<size_t>(blockIdx.x - n_cls_blocks) * kPrepThreads + threadIdx.x) * 8;
        if (i8 >= total) return;
        const float4 x0 = __ldg(reinterpret_cast<const float4 *>(a.q + i8));
        const float4 x1 = __ldg(reinterpret_cast<const float4 *>(a.q + i8) + 1);
        uint4 o;
        if (a.q16_type == kKvBF16) {
            __nv_bfloat162 b0 = __floats2bfloat162_rn(x0.x, x0.y), b1 = __floats2bfloat162_rn(x0.z, x0.w);
            __nv_bfloat162 b2 = __floats2bfloat162_rn(x1.x, x1.y), b3 = __floats2bfloat162_rn(x1.z, x1.w);
            o = make_uint4(*reinterpret_cast<uint32_t *>(&b0), *reinterpret_cast<uint32_t *>(&b1),
                           *reinterpret_cast<uint32_t *>(&b2), *reinterpret_cast<uint32_t *>(&b3));
        } else {
            __half2 h0 = __floats2half2_rn(x0.x, x0.y), h1 = __floats2half2_rn(x0.z, x0.w);
            __half2 h2 = __floats2half2_rn(x1.x, x1.y), h3 = __floats2half2_rn(x1.z, x1.w);
            o = make_uint4(*reinterpret_cast<uint32_t *>(&h0), *reinterpret_cast<uint32_t *>(&h1),
                           *reinterpret_cast<uint32_t *>(&h2), *reinterpret_cast<uint32_t *>(&h3));
        }
        *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.q16) + i8) = o;
        return;
    }
    __shared__ int s_any[kPrepThreads / 32], s_all[kPrepThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int chunk = blockIdx.x;
    const int key = chunk * 32 + lane;
    const bool valid = key < a.N;
    bool any_att = false, all_zero = true;
    if (valid) {
        if (a.mask != nullptr) {
            const float *col = a.mask + key;
#pragma unroll 4
            for (int i = warp; i < a.L; i += kPrepThreads / 32) {
                const float m = __ldg(col + static_cast<size_t>(i) * a.stride);
                any_att |= m > kMasked;
                all_zero &= m == 0.0f;
            }
        } else {
            // implicit causal: row i attends [window_start, N - L + i]
            const int last = a.N - a.L;            // row 0's last attended key
            for (int i = warp; i < a.L; i += kPrepThreads / 32) {
                const bool att = key >= a.window_start && key <= last + i;
                any_att |= att;
                all_zero &= att;
            }
        }
    }
    any_att = __any_sync(0xffffffffu, any_att);
    all_zero = __all_sync(0xffffffffu, all_zero);
    if (lane == 0) { s_any[warp] = any_att; s_all[warp] = all_zero; }
    __syncthreads();
    if (threadIdx.x == 0) {
        bool an = false, al = true;
        for (int w = 0; w < kPrepThreads / 32; ++w) { an |= s_any[w] != 0; al &= s_all[w] != 0; }
        a.cls[chunk] = !an ? kChunkDead : (al ? kChunkAllAttended : kChunkMixed);
    }
}

cudaError_t launch_tree_classify(const TreeArgs &a, cudaStream_t s) {
    const int n_cls = a.n_chunks;
    int n_q = 0;
    if (a.q16_type >= 0) {
        const size_t total = static_cast<size_t>(a.H) * a.L * a.D;
        n_q = static_cast<int>((total + kQ16PerBlock - 1) / kQ16PerBlock);
    }
    cudaError_t e = launch_pdl(tree_prep_kernel, dim3(n_cls + n_q), dim3(kPrepThreads), 0, s, a, n_cls);
    count_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Merge: one CTA per output row (rid = i * H + h) over the partial slots the
// main pass left (workspace header; 0 = the output is already final).  M* and the per-split
// weights e^(M_w - M*) are computed once per row into shared memory (128
// splits at a time); every thread then accumulates its float4 of O over the
// splits with independent loads.
__global__ void __launch_bounds__(128) tree_reduce_kernel(const TreeArgs a) {
    pdl_wait();
    const int nwg = a.err[1];
    if (nwg <= 0) return;
    __shared__ float s_e[128], s_se[128];
    __shared__ float s_red[2];
    const int rid = blockIdx.x;
    const int nrows = a.H * a.L;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int D4 = a.D / 4;
    const float *ml = a.part_ml + static_cast<size_t>(rid) * 2;
    const size_t ml_stride = static_cast<size_t>(nrows) * 2;
    if (warp == 0) {
        float m = -FLT_MAX;
        for (int w = lane; w < nwg; w += 32) m = fmaxf(m, __ldg(ml + w * ml_stride + 1));
        m = warp_max(m);
        if (lane == 0) s_red[0] = m;
    }
    __syncthreads();
    const float mstar = s_red[0];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float ssum = 0.0f;
    const float *po = a.part_o + static_cast<size_t>(rid) * a.D + 4 * t;
    const size_t po_stride = static_cast<size_t>(nrows) * a.D;
    for (int w0 = 0; w0 < nwg; w0 += 128) {
        const int n = min(128, nwg - w0);
        if (t < n) {
            const float e = expf(__ldg(ml + (w0 + t) * ml_stride + 1) - mstar);
            s_e[t] = e;
            s_se[t] = __ldg(ml + (w0 + t) * ml_stride) * e;
        }
        __syncthreads();
        if (t < D4) {
#pragma unroll 4
            for (int j = 0; j < n; ++j) {
                const float4 o = __ldg(reinterpret_cast<const float4 *>(po + (w0 + j) * po_stride));
                const float e = s_e[j];
                acc.x += o.x * e; acc.y += o.y * e; acc.z += o.z * e; acc.w += o.w * e;
            }
        }
        if (warp == 0)
            for (int j = lane; j < n; j += 32) ssum += s_se[j];
        __syncthreads();
    }
    if (warp == 0) {
        ssum = warp_sum(ssum);
        if (lane == 0) s_red[1] = ssum;
    }
    __syncthreads();
    const float sstar = s_red[1];
    const float inv = (sstar == 0.0f) ? 0.0f : 1.0f / sstar;
    if (t < D4) {
        const float4 r = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        reinterpret_cast<float4 *>(a.out + static_cast<size_t>(rid) * a.D)[t] = r;
    }
}

cudaError_t launch_tree_reduce(const TreeArgs &a, cudaStream_t s) {
    cudaError_t e = launch_pdl(tree_reduce_kernel, dim3(a.H * a.L), dim3(128), 0, s, a);
    count_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace ta
