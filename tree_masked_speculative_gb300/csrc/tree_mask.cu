// Dense tree mask from a parent array on the device (the step before the
// verify pass).  The draft tree's node i sits at KV position
// kv_seq_len - q_l + i and attends the prefix [0, kv_seq_len - q_l), its
// ancestors and itself (tree_attention.metal header comment; tree_attention.rs
// tests: 0 = attend, -65504 = masked).  Cells at positions >= kv_seq_len, up
// to mask_stride, are masked too.
//
// Grid (column chunks, q_l): each CTA loads the whole parent array into shared
// memory, walks its row's ancestor chain there (the chain ends at a value
// outside [0, current node), -1 for the root) into a shared bitset, and writes
// its chunk of the row with 16-byte stores when the row is 16-byte aligned.
#include "ta_internal.cuh"

namespace ta {

namespace {

constexpr int kMaskThreads = 256;
constexpr int kMaskChunk = 4096;   // columns per CTA

__global__ void __launch_bounds__(kMaskThreads) tree_mask_kernel(const int32_t *parents, int q_l, int kv_seq_len,
                                                                 int stride, float *mask) {
    extern __shared__ int32_t s_par[];                              // [q_l] parents, then the bitset
    uint32_t *s_anc = reinterpret_cast<uint32_t *>(s_par + q_l);   // [(q_l + 31) / 32]
    const int i = blockIdx.y;
    const int nwords = (q_l + 31) / 32;
    for (int k = threadIdx.x; k < q_l; k += kMaskThreads) s_par[k] = __ldg(parents + k);
    for (int k = threadIdx.x; k < nwords; k += kMaskThreads) s_anc[k] = 0u;
    __syncthreads();
    if (threadIdx.x == 0) {
        int node = i;
        s_anc[node >> 5] |= 1u << (node & 31);
        for (;;) {                                   // at most i steps: each step goes to a smaller node
            const int up = s_par[node];
            if (up < 0 || up >= node) break;
            s_anc[up >> 5] |= 1u << (up & 31);
            node = up;
        }
    }
    __syncthreads();
    const int prefix = kv_seq_len - q_l;
    const int j0 = blockIdx.x * kMaskChunk;
    const int j1 = min(stride, j0 + kMaskChunk);
    float *row = mask + static_cast<size_t>(i) * stride;
    auto cell = [&](int j) -> float {
        if (j < prefix) return 0.0f;
        if (j >= kv_seq_len) return kMasked;
        const int a = j - prefix;
        return (s_anc[a >> 5] >> (a & 31)) & 1u ? 0.0f : kMasked;
    };
    if ((stride & 3) == 0 && (reinterpret_cast<uintptr_t>(mask) & 15u) == 0) {
        for (int j = j0 + 4 * threadIdx.x; j < j1; j += 4 * kMaskThreads)
            *reinterpret_cast<float4 *>(row + j) = make_float4(cell(j), cell(j + 1), cell(j + 2), cell(j + 3));
    } else {
        for (int j = j0 + threadIdx.x; j < j1; j += kMaskThreads) row[j] = cell(j);
    }
}

}  // namespace

cudaError_t launch_tree_mask(const int32_t *parents, int q_l, int kv_seq_len, int stride, float *mask,
                             cudaStream_t s) {
    const size_t smem = sizeof(int32_t) * (static_cast<size_t>(q_l) + (q_l + 31) / 32);
    static unsigned long long done = 0;
    cudaError_t e = set_smem_limit_once(tree_mask_kernel, kMaxTreeMaskSmem, &done);
    if (e != cudaSuccess) return e;
    dim3 grid((stride + kMaskChunk - 1) / kMaskChunk, q_l);
    tree_mask_kernel<<<grid, kMaskThreads, smem, s>>>(parents, q_l, kv_seq_len, stride, mask);
    count_launch();
    return cudaGetLastError();
}

}  // namespace ta
