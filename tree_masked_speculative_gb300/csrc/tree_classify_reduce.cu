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

// Prep pass, one launch: blocks [0, n_cls) classify the chunks, one warp per
// chunk (dead if no (row, key < N) cell is attended (> -65504), all-attended if
// every (row, key < N) cell equals 0.0, else mixed); the remaining blocks
// write the 16-bit copy of Q for the tensor-core kernel; block 0 clears the
// error word.
constexpr int kPrepThreads = 256;
constexpr int kQ16PerBlock = kPrepThreads * 8;

__global__ void __launch_bounds__(kPrepThreads) tree_prep_kernel(const TreeArgs a, int n_cls_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && a.err != nullptr) *a.err = 0;
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
    const int lane = threadIdx.x & 31;
    const int chunk = blockIdx.x * (kPrepThreads / 32) + (threadIdx.x >> 5);
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
    const int n_cls = (a.n_chunks + kPrepThreads / 32 - 1) / (kPrepThreads / 32);
    int n_q = 0;
    if (a.q16_type >= 0) {
        const size_t total = static_cast<size_t>(a.H) * a.L * a.D;
        n_q = static_cast<int>((total + kQ16PerBlock - 1) / kQ16PerBlock);
    }
    tree_prep_kernel<<<n_cls + n_q, kPrepThreads, 0, s>>>(a, n_cls);
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
