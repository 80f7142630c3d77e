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

// One warp per chunk.  Class: dead if no (row, key < N) cell is attended
// (> -65504), all-attended if every (row, key < N) cell equals 0.0, else mixed.
__global__ void __launch_bounds__(256) tree_classify_kernel(const TreeArgs a) {
    const int lane = threadIdx.x & 31;
    const int chunk = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (chunk >= a.n_chunks) return;
    const int key = chunk * 32 + lane;
    const bool valid = key < a.N;
    bool any_att = false, all_zero = true;
    if (valid) {
        if (a.mask != nullptr) {
            const float *col = a.mask + key;
            for (int i = 0; i < a.L; ++i) {
                float m = __ldg(col + (size_t)i * a.stride);
                any_att |= m > kMasked;
                all_zero &= m == 0.0f;
            }
        } else {
            // implicit causal: row i attends [window_start, N - L + i]
            const int last = a.N - a.L;            // row 0's last attended key
            for (int i = 0; i < a.L; ++i) {
                bool att = key >= a.window_start && key <= last + i;
                any_att |= att;
                all_zero &= att;
            }
        }
    }
    any_att = __any_sync(0xffffffffu, any_att);
    all_zero = __all_sync(0xffffffffu, all_zero);
    if (lane == 0) {
        uint8_t cl = !any_att ? kChunkDead : (all_zero ? kChunkAllAttended : kChunkMixed);
        a.cls[chunk] = cl;
    }
}

cudaError_t launch_tree_classify(const TreeArgs &a, cudaStream_t s) {
    dim3 grid((a.n_chunks + 7) / 8);
    tree_classify_kernel<<<grid, 256, 0, s>>>(a);
    count_launch();
    return cudaGetLastError();
}

// One CTA per output row (rid = i * H + h), D/4 threads, float4 per thread.
__global__ void __launch_bounds__(128) tree_reduce_kernel(const TreeArgs a) {
    const int rid = blockIdx.x;
    const int nrows = a.H * a.L;
    const int t = threadIdx.x;              // float4 column
    const int D4 = a.D / 4;
    float mstar = -FLT_MAX;
    for (int w = 0; w < a.nwg; ++w)
        mstar = fmaxf(mstar, __ldg(a.part_ml + ((size_t)w * nrows + rid) * 2 + 1));
    float sstar = 0.0f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int w = 0; w < a.nwg; ++w) {
        const float sw = __ldg(a.part_ml + ((size_t)w * nrows + rid) * 2 + 0);
        const float mw = __ldg(a.part_ml + ((size_t)w * nrows + rid) * 2 + 1);
        const float e = expf(mw - mstar);
        sstar += sw * e;
        if (t < D4) {
            float4 o = __ldg(reinterpret_cast<const float4 *>(a.part_o + ((size_t)w * nrows + rid) * a.D) + t);
            acc.x += o.x * e; acc.y += o.y * e; acc.z += o.z * e; acc.w += o.w * e;
        }
    }
    const float inv = (sstar == 0.0f) ? 0.0f : 1.0f / sstar;
    if (t < D4) {
        float4 r = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        reinterpret_cast<float4 *>(a.out + (size_t)rid * a.D)[t] = r;
    }
}

cudaError_t launch_tree_reduce(const TreeArgs &a, cudaStream_t s) {
    dim3 grid(a.H * a.L);
    tree_reduce_kernel<<<grid, a.D / 4, 0, s>>>(a);
    count_launch();
    return cudaGetLastError();
}

}  // namespace ta
