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

// Classification of one chunk for a tree mask given as a parent array (and,
// by the last chunk's block, the per-row ancestor bitsets the main pass
// reads).  The cells are those of the dense builder: row i attends the prefix
// [0, N - L) and the tree positions N - L + a of itself and its ancestors.  A
// chunk wholly in the prefix is all-attended; a chunk over tree positions
// first builds every row's bitset in shared memory - thread i walks node i's
// chain i, parents[i], ..., which a value outside [0, current node) ends -
// and classifies from it.
static_assert(kPrepThreads >= kMaxTreeBitsNodes, "one thread per tree node");

__device__ __forceinline__ void classify_parents(const TreeArgs &a, int chunk) {
    __shared__ int32_t s_par[kMaxTreeBitsNodes];
    __shared__ uint32_t s_bits[kMaxTreeBitsNodes * (kMaxTreeBitsNodes / 32)];
    __shared__ int s_any[kPrepThreads / 32], s_all[kPrepThreads / 32];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int prefix = a.N - a.L, W = a.anc_words;
    if (chunk * 32 + 32 <= prefix) {
        if (t == 0) a.cls[chunk] = kChunkAllAttended;
        return;
    }
    if (t < a.L) s_par[t] = __ldg(a.parents + t);
    __syncthreads();
    if (t < a.L) {
        uint32_t *row = s_bits + t * W;
        for (int k = 0; k < W; ++k) row[k] = 0u;
        row[t >> 5] |= 1u << (t & 31);
        for (int node = t;;) {                     // at most t steps: each goes to a smaller node
            const int up = s_par[node];
            if (up < 0 || up >= node) break;
            row[up >> 5] |= 1u << (up & 31);
            node = up;
        }
    }
    __syncthreads();
    if (chunk == a.n_chunks - 1)                    // one block publishes the bitsets
        for (int k = t; k < a.L * W; k += kPrepThreads) const_cast<uint32_t *>(a.anc)[k] = s_bits[k];
    const int key = chunk * 32 + lane;
    bool any_att = false, all_zero = true;
    if (key < a.N) {
        const int rel = key - prefix;
        for (int i = warp; i < a.L; i += kPrepThreads / 32) {
            const bool att = rel < 0 || ((s_bits[i * W + (rel >> 5)] >> (rel & 31)) & 1u);
            any_att |= att;
            all_zero &= att;
        }
    }
    any_att = __any_sync(0xffffffffu, any_att);
    all_zero = __all_sync(0xffffffffu, all_zero);
    if (lane == 0) { s_any[warp] = any_att; s_all[warp] = all_zero; }
    __syncthreads();
    if (t == 0) {
        bool an = false, al = true;
        for (int w = 0; w < kPrepThreads / 32; ++w) { an |= s_any[w] != 0; al &= s_all[w] != 0; }
        a.cls[chunk] = !an ? kChunkDead : (al ? kChunkAllAttended : kChunkMixed);
    }
}

__device__ __forceinline__ void prep_body(const TreeArgs &a, int n_cls_blocks) {
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
    if (a.anc != nullptr) {
        classify_parents(a, static_cast<int>(blockIdx.x));
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

// Launched as a programmatic dependent: the main pass that follows may start
// launching at once (it waits for this grid), and this grid waits for its own
// predecessor - the previous merge, or whatever kernel wrote Q and the mask -
// before it reads anything or touches the workspace.
__global__ void __launch_bounds__(kPrepThreads) tree_prep_kernel(const TreeArgs a, int n_cls_blocks) {
    pdl_launch_dependents();
    pdl_wait();
    prep_body(a, n_cls_blocks);
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
// main pass left (workspace header; 0 = the output is already final).  Thread
// t takes float4 column (t % D4) of the slots w = t / D4 (mod groups): all its
// (S, M) and O loads are issued together and merged against the thread's own
// running max; the groups are then combined in shared memory with the
// log-sum-exp weights e^(m_g - M*).  One round trip to memory.
constexpr int kReduceThreads = 256;

__global__ void __launch_bounds__(kReduceThreads) tree_reduce_kernel(const TreeArgs a) {
    pdl_wait();
    // The next prep pass may start launching; it waits for this grid to finish
    // before it rewrites the workspace.
    pdl_launch_dependents();
    __shared__ float4 s_acc[kReduceThreads];
    __shared__ float2 s_ms[kReduceThreads];   // (m_g, s_g) per thread
    const int rid = blockIdx.x;
    const int nrows = a.H * a.L;
    const int t = threadIdx.x;
    const int D4 = a.D / 4;
    const int groups = kReduceThreads / D4;
    const int g = t / D4, i = t % D4;
    const float2 *ml = reinterpret_cast<const float2 *>(a.part_ml) + rid;   // (S, M), stride nrows
    const float *po = a.part_o + static_cast<size_t>(rid) * a.D + 4 * i;
    const size_t po_stride = static_cast<size_t>(nrows) * a.D;
    // The thread's first kPre slots (of the a.nwg the workspace holds) are
    // loaded together with the slot count the main pass published, so the
    // count costs no round trip of its own; slots past the count are ignored.
    constexpr int kPre = 4;
    float2 sm_pre[kPre];
    float4 o_pre[kPre];
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
        const int w = g + k * groups;
        if (g < groups && w < a.nwg) {
            sm_pre[k] = __ldg(ml + static_cast<size_t>(w) * nrows);
            o_pre[k] = __ldg(reinterpret_cast<const float4 *>(po + w * po_stride));
        }
    }
    const int nwg = a.err[1];
    if (nwg <= 0) return;
    float m = -FLT_MAX, ssum = 0.0f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    auto merge = [&](float2 sm, float4 o) {
        // a slot with no attended key (S = 0) adds nothing; its O is not read
        // (slots that no split fills are marked this way and left unwritten)
        if (sm.x == 0.0f) return;
        const float mn = fmaxf(m, sm.y);
        const float c = expf(m - mn), e = expf(sm.y - mn);
        m = mn;
        ssum = ssum * c + sm.x * e;
        acc.x = acc.x * c + o.x * e; acc.y = acc.y * c + o.y * e;
        acc.z = acc.z * c + o.z * e; acc.w = acc.w * c + o.w * e;
    };
    if (g < groups) {
#pragma unroll
        for (int k = 0; k < kPre; ++k)
            if (g + k * groups < nwg) merge(sm_pre[k], o_pre[k]);
#pragma unroll 4
        for (int w = g + kPre * groups; w < nwg; w += groups)
            merge(__ldg(ml + static_cast<size_t>(w) * nrows),
                  __ldg(reinterpret_cast<const float4 *>(po + w * po_stride)));
    }
    s_acc[t] = acc;
    s_ms[t] = make_float2(m, ssum);
    __syncthreads();
    if (t < D4) {
        float mstar = -FLT_MAX;
        for (int k = 0; k < groups; ++k) mstar = fmaxf(mstar, s_ms[k * D4 + t].x);
        float sstar = 0.0f;
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = 0; k < groups; ++k) {
            const float2 ms = s_ms[k * D4 + t];
            const float w = expf(ms.x - mstar);
            const float4 x = s_acc[k * D4 + t];
            sstar += ms.y * w;
            r.x += x.x * w; r.y += x.y * w; r.z += x.z * w; r.w += x.w * w;
        }
        const float inv = (sstar == 0.0f) ? 0.0f : 1.0f / sstar;
        reinterpret_cast<float4 *>(a.out + static_cast<size_t>(rid) * a.D)[t] =
            make_float4(r.x * inv, r.y * inv, r.z * inv, r.w * inv);
    }
}

cudaError_t launch_tree_reduce(const TreeArgs &a, cudaStream_t s) {
    cudaError_t e = launch_pdl(tree_reduce_kernel, dim3(a.H * a.L), dim3(kReduceThreads), 0, s, a);
    count_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace ta
