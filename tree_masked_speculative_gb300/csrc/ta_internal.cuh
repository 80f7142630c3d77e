// Internal declarations of the tree-verify attention library (not installed).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cfloat>

namespace ta {

// Sentinel of a masked tree-mask cell (-MAXHALF), and the running-max start
// value of the online softmax (mlx-native tree_attention.metal, main kernel).
constexpr float kMasked = -65504.0f;
constexpr float kMInit = -FLT_MAX / 2;

// Chunk classes written by the mask-compaction pass, one byte per 32 keys.
enum ChunkClass : uint8_t { kChunkDead = 0, kChunkAllAttended = 1, kChunkMixed = 2 };

// Largest draft tree (q_l) whose mask may be given as a parent array: its
// per-row ancestor bitsets ((q_l + 31) / 32 words a row) live in the workspace.
constexpr int kMaxTreeBitsNodes = 256;

enum KvType : int { kKvF32 = 0, kKvF16 = 1, kKvBF16 = 2 };

// ------------------------------------------------------------ device helpers
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Programmatic dependent launch: a kernel launched with launch_pdl() may start
// while its predecessor in the stream still runs; pdl_wait() blocks until the
// predecessor has completed and its writes are visible.  launch_dependents()
// lets the next such kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Expand one 16-byte vector of KV_T into floats.
template <typename KV_T>
struct Vec16;
template <>
struct Vec16<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void expand(const uint4 &u, float *f) {
        f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
    }
};
template <>
struct Vec16<__half> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void expand(const uint4 &u, float *f) {
        const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) { float2 t = __half22float2(h[i]); f[2 * i] = t.x; f[2 * i + 1] = t.y; }
    }
};
template <>
struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void expand(const uint4 &u, float *f) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};

// ------------------------------------------------------------------- args
struct TreeArgs {
    const float *q;        // [H, L, D] f32
    const void *k;         // [Hk, C, D] KV_T
    const void *v;
    const float *mask;     // [L, stride] f32; nullptr (and no anc) -> implicit causal
    const uint32_t *anc;   // [L][anc_words] ancestor bitsets of a parent array (written by
                           // the prep pass), or nullptr
    const int32_t *parents;  // [L] the parent array (device), with anc
    int anc_words;         // (L + 31) / 32
    uint8_t *cls;          // [n_chunks] chunk classes
    float *part_o;         // [nwg][nrows][D]
    float *part_ml;        // [nwg][nrows][2] = (S, M)
    float *out;            // [L, H, D]
    void *q16;             // [H*L, D] 16-bit copy of Q (tensor-core path)
    int *err;              // workspace error word (0 = ok), zeroed by the prep pass
    int H, Hk, D, N, C, L, stride, nwg, g, R, n_chunks, window_start;
    int q16_type;          // -1: no 16-bit Q copy, else kKvF16 / kKvBF16
    int n_part;            // partial slots the main pass leaves for the merge (0 = output final)
    int cluster_x;         // tensor-core kernel: splits merged inside one cluster
    int flat_groups;       // CTA pairs: groups per O half of the flattened schedule (0 = uniform splits)
    float scale;
};

// Cell (query row qi, key < N) of an explicit tree mask: the dense mask row
// `mrow`, or, when the mask came as a parent array, 0 on the prefix
// [0, N - L) and at the tree positions N - L + a for a in qi's ancestor
// bitset (itself included), -65504 elsewhere - the cells tree_mask_build
// writes for the same parents.
__device__ __forceinline__ float explicit_cell(const TreeArgs &a, const float *mrow, int qi, int key) {
    if (a.anc == nullptr) return __ldg(mrow + key);
    const int rel = key - (a.N - a.L);
    if (rel < 0) return 0.0f;
    const uint32_t w = __ldg(a.anc + static_cast<size_t>(qi) * a.anc_words + (rel >> 5));
    return ((w >> (rel & 31)) & 1u) ? 0.0f : kMasked;
}

// The 32 explicit-mask cells of row qi for keys key0 .. key0 + 31 (masked at
// keys >= N), the mask's kind decided once for the chunk.
__device__ __forceinline__ void explicit_chunk(const TreeArgs &a, const float *mrow, int qi, int key0,
                                               float (&x)[32]) {
    if (a.anc == nullptr) {
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = key0 + e < a.N ? __ldg(mrow + key0 + e) : kMasked;
    } else {
        // the chunk's tree positions span at most two bitset words of the row
        const int rel0 = key0 - (a.N - a.L);
        const uint32_t *row = a.anc + static_cast<size_t>(qi) * a.anc_words;
        const int w0 = rel0 >> 5;   // arithmetic shift: -1 for a chunk that starts in the prefix
        const uint32_t lo = w0 >= 0 && w0 < a.anc_words ? __ldg(row + w0) : 0u;
        const uint32_t hi = w0 + 1 >= 0 && w0 + 1 < a.anc_words ? __ldg(row + w0 + 1) : 0u;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const int rel = rel0 + e;
            const uint32_t w = (rel >> 5) == w0 ? lo : hi;
            x[e] = key0 + e >= a.N ? kMasked : (rel < 0 ? 0.0f : (((w >> (rel & 31)) & 1u) ? 0.0f : kMasked));
        }
    }
}

// TMA descriptors of the tensor-core tree kernel (kernel parameters).
struct TcMaps {
    CUtensorMap q16;   // 2D {D, H*L} 16-bit, box {64, 128}, 128-byte swizzle
    CUtensorMap k;     // 3D {D, kv_seq_len, Hk}, box {64, 32, 1}, 128-byte swizzle (one chunk)
    CUtensorMap v;
    CUtensorMap k64;   // the same tensors, box {64, 64, 1}: two consecutive chunks (CTA pairs)
    CUtensorMap v64;
};

struct QuantArgs {
    const void *queries;     // [B*nQ, dim] T
    const uint32_t *kp, *vp; // [B*nKV, N, wpt]
    const void *ks, *kb, *vs, *vb;  // [B*nKV, N, ng] T
    const float *sinks;      // [nQ]
    const uint32_t *mbool;   // [B*nQ, N] or nullptr
    const void *mfloat;      // [B*nQ, N] T or nullptr
    float *part_o;           // [nwg][rows][dim]
    float *part_ml;          // [nwg][rows][2] = (S, M), M in log2 units
    void *out;               // [rows, dim] T or f32
    int rows, nQ, rep, kv_rows, dim, N, bits, G, has_sinks, window, nwg;
    int wpt, ng;             // packed words and scale groups per token
    int n_rg;                // row groups of kQuantRowsPerCta query rows per KV row
    int t_lo;                // first token of the window
    int c_lo, nch;           // first chunk of the window, chunks per KV row
    int al_sb;               // scale/bias chunks start on 16-byte boundaries
    int al_mb;               // bool-mask chunks start on 16-byte boundaries
    int al_mf;               // float-mask chunks start on 16-byte boundaries
    int *err;                // error word (bit 0: a copy wait timed out), never cleared here
    uint32_t first_wait_polls;   // CUDA-core kernel: bound of each CTA's first copy wait
    const int32_t *tree_parents; // [tree_ql] parent array of a draft tree over the last tree_ql tokens, or nullptr
    int tree_ql;                 // 0: no tree mask; else row q is node q % tree_ql of that tree
    int t_is_bf16, out_f32;
    float scale;
    // tensor-core kernel only: rows per CTA (4, 8, 16 or 32), row blocks per KV row,
    // first 128-token tile and tile count of the window, ring depths (decoded
    // chunks, packed-K slots, packed-V slots) and TMEM columns
    int rp, n_rb, j_lo, ntile, tc_nd, tc_nk, tc_nv, tc_cols;
};

// Largest draft tree a quantized-KV call takes as a parent array (one 32-bit
// ancestor bitset per node).
constexpr int kMaxQuantTreeNodes = 32;

// Ancestor bitset of node `lane` (lane < L <= 32; 0 for the other lanes):
// the node itself and the chain lane, parents[lane], ... that a value outside
// [0, current node) ends (the rule of tree_mask_build).  Warp-collective: lane
// i holds parents[i] and the chains are followed by shuffles, one level per
// step, so no chain waits on a dependent global load.
// `up` is parents[lane] (any value for lane >= L), loaded by the caller.
__device__ __forceinline__ uint32_t quant_tree_ancestors(int up, int L) {
    const int lane = static_cast<int>(threadIdx.x & 31u);
    if (lane >= L || up < 0 || up >= lane) up = -1;        // the chain ends at this node
    uint32_t bits = lane < L ? 1u << lane : 0u;
    int node = lane < L ? up : -1;
    for (int step = 0; step < L; ++step) {                 // each step goes to a smaller node
        if (node >= 0) bits |= 1u << node;
        const int nxt = __shfl_sync(0xffffffffu, up, node >= 0 ? node : 0);
        node = node >= 0 ? nxt : -1;
    }
    return bits;
}

// Bound (polls) of every mbarrier wait of the CUDA-core quantized-KV kernel.
constexpr uint32_t kQuantWaitPolls = 1u << 22;
// Query rows served by one CTA of the quantized-KV kernel (a row group).
constexpr int kQuantRowsPerCta = 4;
// Dynamic shared-memory limit requested for the quantized-KV kernels.
constexpr size_t kQuantMaxSmem = 227 * 1024;
// Bytes at the start of the quantized path's tmp buffer holding its error
// word (the split partials follow).
constexpr size_t kQuantErrBytes = 256;

// Per-warp shared-memory layout of the quantized-KV kernel (byte offsets,
// 16-aligned).  Group A of a chunk (packed K words, raw scale / bias copies,
// bool and float mask rows) and group B (packed V words) are double-buffered;
// then the scales as {s, s, -2^23 s, -2^23 s}, the weights {p, p} per
// (token, row), the per-lane V-bias accumulators, the q-group sums and four
// mbarriers.
struct QuantLayout {
    int a0, a_stage;                    // group-A stage b at a0 + b * a_stage
    int k, ks, kb, vs, vb, mb, mf;      // offsets inside a group-A stage
    int v0, v_stage;                    // group-B stage b at v0 + b * v_stage
    int ks4, vs4, p2, ob, qs, bars, total;
};
__host__ __device__ inline int quant_take(int *o, int bytes) {
    const int r = *o;
    *o += (bytes + 15) & ~15;
    return r;
}
// ns: stages of each group (the CUDA-core kernel uses two); rows: query rows
// whose mask rows a stage holds.
__host__ __device__ inline QuantLayout quant_layout(int wpt, int ng, int ch, int ns = 2,
                                                    int rows = kQuantRowsPerCta) {
    const int R = rows;
    QuantLayout L;
    int o = 0;   // inside a group-A stage
    L.k = quant_take(&o, ch * wpt * 4);
    L.ks = quant_take(&o, ch * ng * 2);
    L.kb = quant_take(&o, ch * ng * 2);
    L.vs = quant_take(&o, ch * ng * 2);
    L.vb = quant_take(&o, ch * ng * 2);
    L.mb = quant_take(&o, R * ch * 4);
    L.mf = quant_take(&o, R * ch * 2);
    L.a_stage = o;
    o = 0;
    L.a0 = quant_take(&o, ns * L.a_stage);
    L.v_stage = (ch * wpt * 4 + 15) & ~15;
    L.v0 = quant_take(&o, ns * L.v_stage);
    L.ks4 = quant_take(&o, ch * ng * 16);
    L.vs4 = quant_take(&o, ch * ng * 16);
    L.p2 = quant_take(&o, (ch > 32 ? ch : 32) * R * 8);   // also holds [row][32] q sums
    L.ob = quant_take(&o, 32 * ng * 4);
    L.qs = quant_take(&o, R * ng * 4);
    L.bars = quant_take(&o, 4 * 8);
    L.total = o;
    return L;
}
// Shared-memory layout of the tensor-core quantized-KV kernel (byte offsets).
// Two P buffers (the PV operand P^T: [rp rows][128 tokens] 16-bit, 128-byte
// swizzled, two 64-token k-blocks of rp * 128 bytes for P_hi, then two for
// P_lo; rows past the CTA's
// query rows are never written and only feed O^T columns that are never
// read), the 16-bit Q operand ([rp][dim], 64-dimension blocks), the ring of
// decoded 16 KB chunks ([128 tokens][64 dims] f16: K half, V half), the
// packed-K ring, the packed-V ring (V words, K and V scale / bias runs, bool
// and float mask rows), per-row constants, the softmax exchange area and the
// mbarriers.
struct QtcLayout {
    int pkb;                              // bytes of a 64-token k-block of a P buffer (rp x 128 B)
    int p0, q0, d0, k0, kslot, v0, vslot;
    int vw, vks, vkb, vvs, vvb, vmb, vmf;  // inside a packed-V slot
    int rc, red, bars, total;
};
constexpr int kQtcChunk = 16384;
constexpr int kQuantTcMaxRing = 16;   // deepest ring of the tensor-core quantized kernel
constexpr int kQtcRedBytes = 4096;   // softmax exchange area (row maxima, row sums, final maxima)
constexpr int kQtcBarBytes = 1280;
__host__ __device__ inline int qtc_align(int o, int a) { return (o + a - 1) / a * a; }
__host__ __device__ inline QtcLayout qtc_layout(int rp, int dim, int wpt, int ng, int nd, int nk, int nv,
                                                bool has_mb, bool has_mf) {
    QtcLayout L;
    L.pkb = rp * 128;
    int o = 0;
    L.p0 = o;
    o += 8 * L.pkb;
    o = qtc_align(o, 1024);
    L.q0 = o;
    o += (dim / 64) * rp * 128;
    o = qtc_align(o, 1024);
    L.d0 = o;
    o += nd * kQtcChunk;
    // a 64-dimension V chunk is read as the first half of a 128-dimension MMA
    // operand: keep the chunk-sized read past the ring inside the allocation
    if (dim < 128) o += kQtcChunk;
    L.kslot = qtc_align(128 * wpt * 4, 16);
    L.k0 = o;
    o += nk * L.kslot;
    int v = 0;
    L.vw = v;  v = qtc_align(v + 128 * wpt * 4, 16);
    L.vks = v; v = qtc_align(v + 128 * ng * 2, 16);
    L.vkb = v; v = qtc_align(v + 128 * ng * 2, 16);
    L.vvs = v; v = qtc_align(v + 128 * ng * 2, 16);
    L.vvb = v; v = qtc_align(v + 128 * ng * 2, 16);
    L.vmb = v; if (has_mb) v = qtc_align(v + rp * 128 * 4, 16);
    L.vmf = v; if (has_mf) v = qtc_align(v + rp * 128 * 2, 16);
    L.vslot = v;
    L.v0 = o;
    o += nv * L.vslot;
    L.rc = o;
    o = qtc_align(o + (rp + ng * rp) * 4, 16);
    L.red = o;
    o = qtc_align(o + kQtcRedBytes, 16);
    o = qtc_align(o, 8);
    L.bars = o;
    o += kQtcBarBytes;
    L.total = o;
    return L;
}

// Head-dimension capacity of the kernel instance serving `dim` (64..512), and
// its chunk length in tokens (32 when a token has at most 32 packed words).
__host__ __device__ inline int quant_dim_capacity(int dim) {
    return dim <= 64 ? 64 : (dim <= 128 ? 128 : (dim <= 256 ? 256 : 512));
}
__host__ __device__ inline int quant_chunk_tokens(int dim, int bits) {
    return quant_dim_capacity(dim) * bits / 32 <= 32 ? 32 : 16;
}

// Workspace layout inside the caller's tmp buffer (all offsets 256-aligned).
struct TreeWorkspace {
    size_t off_part_o, off_part_ml, off_cls, off_q16, off_anc, off_err, total;
};

// ------------------------------------------------------------ host launches
// Each returns cudaGetLastError() after enqueueing on `s`.
cudaError_t launch_tree_classify(const TreeArgs &a, cudaStream_t s);
cudaError_t launch_tree_fma(const TreeArgs &a, int kv_type, cudaStream_t s);
cudaError_t launch_tree_tc(const TreeArgs &a, const TcMaps &maps, int kv_type, cudaStream_t s);
// Whether the tensor-core tree kernel runs as CTA pairs (cta_group::2): head
// dimension 512 with more than 128 rows per KV head, where each CTA then
// loads half of every key tile (measured faster there; with D <= 256 the
// one-CTA form is).
__host__ __device__ inline bool tree_tc_pairs(int R, int D) { return R > 128 && D == 512; }
// Row tiles (CTAs along the rows of a KV head) of the tensor-core kernel:
// ceil(R / 128), rounded up to an even count for CTA pairs.
__host__ __device__ inline int tree_tc_row_ctas(int R, int D) {
    const int n_rt = (R + 127) / 128;
    return tree_tc_pairs(R, D) ? 2 * ((n_rt + 1) / 2) : n_rt;
}
// Flattened schedule of the CTA pairs.  Units are (KV head, pair of row
// tiles), each with tpu key tiles of 4 chunks; the U x tpu (unit, tile)
// positions are cut into G contiguous ranges of nearly equal length, one per
// pair-group (per O half), so that every SM gets the same share of work when
// the uniform split count would leave some idle.  A range meets at most two
// units (G >= U); the part in one unit is a segment, which leaves one partial
// slot for the merge: its group's index minus that of the unit's first group.
__host__ __device__ inline long long flat_start(int g, long long W, int G) { return (long long)g * W / G; }
// Group whose range holds position P (0 <= P < W).
__host__ __device__ inline int flat_group_of(long long P, long long W, int G) {
    int g = static_cast<int>(P * G / W);
    while (g + 1 < G && flat_start(g + 1, W, G) <= P) ++g;
    while (g > 0 && flat_start(g, W, G) > P) --g;
    return g;
}
// Partial slots unit u uses.
__host__ __device__ inline int flat_unit_slots(int u, int tpu, long long W, int G) {
    return flat_group_of((long long)(u + 1) * tpu - 1, W, G) - flat_group_of((long long)u * tpu, W, G) + 1;
}
// Cluster shape of the tensor-core kernel: x = splits merged in-cluster (y = 1).
void tree_tc_cluster_shape(const TreeArgs &a, int *cx, int *cy);
cudaError_t launch_tree_reduce(const TreeArgs &a, cudaStream_t s);
// Dense tree mask [q_l, stride] f32 from parents [q_l] (device pointers).
cudaError_t launch_tree_mask(const int32_t *parents, int q_l, int kv_seq_len, int stride, float *mask,
                             cudaStream_t s);
// Largest q_l the mask builder takes (its parents and bitset live in shared memory).
constexpr int kMaxTreeMaskNodes = 16384;
constexpr size_t kMaxTreeMaskSmem = sizeof(int32_t) * (kMaxTreeMaskNodes + kMaxTreeMaskNodes / 32);
cudaError_t launch_quant_fma(const QuantArgs &a, cudaStream_t s);
cudaError_t launch_quant_merge(const QuantArgs &a, cudaStream_t s);
cudaError_t launch_quant_b4(const QuantArgs &a, cudaStream_t s);
cudaError_t launch_quant_b8(const QuantArgs &a, cudaStream_t s);
// Resident CTAs (warps) per SM of the quantized-KV kernel for (bits, dim,
// groups per token); 0 if it cannot be determined.
int quant_ctas_per_sm(int bits, int dim, int ng);
int quant_ctas_per_sm_b4(int dim, int ng);
int quant_ctas_per_sm_b8(int dim, int ng);
// Tensor-core quantized-KV kernel (rows on the N side of the score MMA):
// launch, and resident CTAs per SM for a dynamic shared-memory size.
cudaError_t launch_quant_tc(const QuantArgs &a, size_t smem, cudaStream_t s);
cudaError_t launch_quant_tc_b4(const QuantArgs &a, size_t smem, cudaStream_t s);
cudaError_t launch_quant_tc_b8(const QuantArgs &a, size_t smem, cudaStream_t s);
int quant_tc_ctas_per_sm(int bits, int rp, size_t smem);
int quant_tc_ctas_per_sm_b4(int rp, size_t smem);
int quant_tc_ctas_per_sm_b8(int rp, size_t smem);
// Warp-MMA quantized-KV kernel (mma.sync, one warp per CTA, 4 query rows):
// head dimension 64, 128 or 256 exactly and group size 32 or 64.
bool quant_mma_shape_ok(int dim, int group_size);
// Its wide form (16 query rows per warp, quant_mma16.cuh): from 16 query rows
// per KV row, head dimension 64 or 128, group size 32 or 64.
bool quant_mma_wide(int rep, int dim, int group_size);
// Query rows of one warp-MMA CTA for rep rows per KV row (4, or 16 in the wide form).
int quant_mma_rows(int rep, int dim, int group_size);
// CTAs per SM the two-warp form's split count is sized for (at most).
constexpr int kQmmaTwoWarpCtasPerSm = 6;
cudaError_t launch_quant_mma(const QuantArgs &a, cudaStream_t s);
cudaError_t launch_quant_mma_b4(const QuantArgs &a, cudaStream_t s);
cudaError_t launch_quant_mma_b8(const QuantArgs &a, cudaStream_t s);
cudaError_t launch_quant_mma16_b4(const QuantArgs &a, cudaStream_t s);
cudaError_t launch_quant_mma16_b8(const QuantArgs &a, cudaStream_t s);
int quant_mma_ctas_per_sm(int bits, int dim, int ng, int rep);
int quant_mma_ctas_per_sm_b4(int dim, int ng);
int quant_mma_ctas_per_sm_b8(int dim, int ng);
int quant_mma16_ctas_per_sm_b4(int dim, int ng);
int quant_mma16_ctas_per_sm_b8(int dim, int ng);

// Rows of one CTA in the CUDA-core tree kernel.
constexpr int kFmaRowsPerCta = 16;

void count_launch(int n = 1);

// Set the calling thread's ta_last_error() message (printf format).
void set_last_error(const char *fmt, ...);

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// As launch_pdl, as clusters of cluster_x x cluster_y CTAs (1 x 1 = no cluster).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                               unsigned cluster_x, unsigned cluster_y, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = cluster_y;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cluster_x * cluster_y > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Raise a kernel's dynamic shared-memory limit once per device; later calls
// (for example while a CUDA graph is being captured) only read a flag.
template <typename Kern>
cudaError_t set_smem_limit_once(Kern kern, size_t bytes, unsigned long long *done_mask) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) __atomic_fetch_or(done_mask, bit, __ATOMIC_ACQ_REL);
    return e;
}

}  // namespace ta
