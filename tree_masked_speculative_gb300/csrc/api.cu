// C ABI of the tree-verify attention library: argument checks, workspace
// layout, split-count choice and kernel dispatch.
//
// The checks restate mlx-native tree_attention.rs (validate_params,
// validate_buffers with overflow-checked byte counts, tmp_buffer_bytes with
// saturating arithmetic) for the tree path, and the shape rules of
// metaltile-std flash_quantized_sdpa.rs (module doc "Layout", dispatch
// invariants) for the quantized path.  Every check runs before any launch.
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "ta_internal.cuh"
#include "tree_attn.h"

#define TA_EXPORT extern "C" __attribute__((visibility("default")))

static_assert(sizeof(ta_tree_params) == 36, "ta_tree_params must be 9 x 4 bytes");

namespace ta {
namespace {

thread_local std::string g_err;
std::atomic<uint64_t> g_launches{0};
constexpr int kQuantTcMinRows = 16;  // automatic choice: tensor cores from this many rows per KV row

ta_status fail(ta_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return st;
}

ta_status cuda_fail(cudaError_t e, const char *what) {
    return fail(TA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool mul3(uint64_t a, uint64_t b, uint64_t c, uint64_t *out) {
    uint64_t t;
    if (__builtin_mul_overflow(a, b, &t)) return false;
    return !__builtin_mul_overflow(t, c, out);
}
bool mul4(uint64_t a, uint64_t b, uint64_t c, uint64_t d, uint64_t *out) {
    uint64_t t;
    return mul3(a, b, c, &t) && !__builtin_mul_overflow(t, d, out);
}
uint64_t sat_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    return __builtin_mul_overflow(a, b, &r) ? UINT64_MAX : r;
}
uint64_t align256(uint64_t x) { return (x + 255u) & ~uint64_t(255); }

size_t elt_bytes(int dtype) {
    switch (dtype) {
        case TA_F32: return 4;
        case TA_F16: return 2;
        case TA_BF16: return 2;
        case TA_U32: return 4;
        default: return 0;
    }
}
const char *dtype_name(int dtype) {
    switch (dtype) {
        case TA_F32: return "F32";
        case TA_F16: return "F16";
        case TA_BF16: return "BF16";
        case TA_U32: return "U32";
        case TA_I32: return "I32";
        default: return "unknown";
    }
}

std::atomic<int> g_sm_count[64];   // per device, 0 = not queried yet

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return 0; }
    if (dev >= 0 && dev < 64 && (n = g_sm_count[dev].load(std::memory_order_relaxed)) > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (dev >= 0 && dev < 64) g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

// ---------------------------------------------------------------- tree params
ta_status check_tree_params(const ta_tree_params *p, bool need_mask_stride) {
    if (p == nullptr) return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: params is NULL");
    if (p->head_dim != 128 && p->head_dim != 256 && p->head_dim != 512)
        return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: head_dim must be 128, 256, or 512, got %u",
                    p->head_dim);
    if (p->n_heads == 0 || p->n_kv_heads == 0)
        return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: num_heads and num_kv_heads must be > 0");
    if (p->n_heads % p->n_kv_heads != 0)
        return fail(TA_ERR_INVALID_ARGUMENT,
                    "tree_attention: num_heads (%u) must be divisible by num_kv_heads (%u)", p->n_heads,
                    p->n_kv_heads);
    if (p->kv_seq_len == 0) return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: kv_seq_len must be > 0");
    if (p->kv_capacity < p->kv_seq_len)
        return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: kv_capacity (%u) must be >= kv_seq_len (%u)",
                    p->kv_capacity, p->kv_seq_len);
    if (p->q_l == 0) return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: q_l (q_seq_len) must be > 0");
    if (need_mask_stride && p->mask_stride < p->kv_seq_len)
        return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: mask_stride (%u) must be >= kv_seq_len (%u)",
                    p->mask_stride, p->kv_seq_len);
    // The kernels index with 32-bit ints and launch H * q_l reduce blocks.
    const uint64_t nrows = (uint64_t)p->n_heads * p->q_l;
    if (p->kv_capacity > (uint32_t)INT_MAX || p->mask_stride > (uint32_t)INT_MAX || nrows > (uint64_t)INT_MAX ||
        p->n_kv_heads > 65535u)
        return fail(TA_ERR_UNSUPPORTED, "tree_attention: sizes exceed the kernels' 32-bit index range");
    if (!std::isfinite(p->scale)) return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: scale is not finite");
    return TA_OK;
}

int rows_per_kv(const ta_tree_params *p) { return (int)(p->n_heads / p->n_kv_heads * p->q_l); }

// CTA pairs: groups per O half of the flattened schedule (a group is one pair
// for each O half), or 0 when the pairs are not used, the caller chose nwg,
// or the uniform split count already fills every SM.
int tree_flat_groups(const ta_tree_params *p) {
    if (p->nwg != 0) return 0;
    const int R = static_cast<int>(rows_per_kv(p)), D = static_cast<int>(p->head_dim);
    if (R < 16 || !tree_tc_pairs(R, D)) return 0;
    const int sms = sm_count();
    if (sms <= 0) return 0;
    const int G = sms / 4;
    const int U = static_cast<int>(p->n_kv_heads) * (tree_tc_row_ctas(R, D) / 2);
    const long long tpu = ((static_cast<long long>(p->kv_seq_len) + 31) / 32 + 3) / 4;
    if (U > G || G % U == 0 || static_cast<long long>(U) * tpu < G) return 0;
    return G;
}

uint32_t resolve_tree_nwg(const ta_tree_params *p) {
    if (p->nwg != 0) return p->nwg;
    if (const int G = tree_flat_groups(p)) {
        // partial slots: the most groups any unit's key tiles meet
        const int R = static_cast<int>(rows_per_kv(p)), D = static_cast<int>(p->head_dim);
        const int U = static_cast<int>(p->n_kv_heads) * (tree_tc_row_ctas(R, D) / 2);
        const int tpu = static_cast<int>(((p->kv_seq_len + 31) / 32 + 3) / 4);
        const long long W = static_cast<long long>(U) * tpu;
        int most = 1;
        for (int u = 0; u < U; ++u) most = std::max(most, flat_unit_slots(u, tpu, W, G));
        return static_cast<uint32_t>(most);
    }
    const int sms = sm_count();
    if (sms <= 0) return 0;
    const uint64_t n_chunks = (p->kv_seq_len + 31u) / 32u;
    const uint64_t R = (uint64_t)rows_per_kv(p);
    uint64_t nwg;
    if (R >= 16) {
        // tensor-core kernel: one CTA per SM, CTAs = splits x row tiles x O halves x KV heads
        // and each split a run of whole 4-chunk key tiles (no split gets more tiles
        // than needed to cover the keys with at most one CTA per SM)
        const uint64_t units = (uint64_t)p->n_kv_heads * (uint64_t)tree_tc_row_ctas((int)R, (int)p->head_dim) * (p->head_dim == 512 ? 2 : 1);
        const uint64_t tiles = (n_chunks + 3) / 4;
        uint64_t most = (uint64_t)sms / units;
        if (most < 1) most = 1;
        const uint64_t per_split = (tiles + most - 1) / most;
        nwg = (tiles + per_split - 1) / per_split;
    } else {
        const uint64_t units = (uint64_t)p->n_kv_heads * ((R + kFmaRowsPerCta - 1) / kFmaRowsPerCta);
        nwg = (2ull * sms + units - 1) / units;
        if (nwg > n_chunks) nwg = n_chunks;
    }
    if (nwg < 1) nwg = 1;
    if (nwg > 65535) nwg = 65535;
    return (uint32_t)nwg;
}

bool tree_workspace(const ta_tree_params *p, uint32_t nwg, TreeWorkspace *ws) {
    const uint64_t nrows = (uint64_t)p->n_heads * p->q_l;
    uint64_t po, pml, q16;
    if (!mul4(nwg, nrows, p->head_dim, 4, &po) || !mul4(nwg, nrows, 2, 4, &pml) ||
        !mul3(nrows, p->head_dim, 2, &q16))
        return false;
    ws->off_part_o = 0;
    ws->off_part_ml = po;
    const uint64_t n_chunks = (p->kv_seq_len + 31u) / 32u;
    ws->off_cls = align256(po + pml);
    ws->off_q16 = align256(ws->off_cls + n_chunks);
    // ancestor bitsets of a parent-array tree mask (trees of up to kMaxTreeBitsNodes nodes)
    const uint64_t anc = p->q_l <= (uint32_t)kMaxTreeBitsNodes ? (uint64_t)p->q_l * ((p->q_l + 31u) / 32u) * 4u : 0u;
    ws->off_anc = align256(ws->off_q16 + q16);
    ws->off_err = align256(ws->off_anc + anc);
    ws->total = ws->off_err + 256;
    return ws->total >= ws->off_q16;
}

const ta_buf kAbsent = {nullptr, 0, TA_F32, 0};

// An optional buffer is absent when its descriptor is NULL or {NULL, 0}.
bool absent(const ta_buf *b) { return b == nullptr || (b->ptr == nullptr && b->bytes == 0); }
const ta_buf &deref(const ta_buf *b) { return b ? *b : kAbsent; }

ta_status check_buf(const ta_buf &b, const char *name, uint64_t need_bytes, size_t align) {
    if (b.reserved != 0) return fail(TA_ERR_INVALID_ARGUMENT, "%s: reserved field must be 0", name);
    if (b.ptr == nullptr) return fail(TA_ERR_INVALID_ARGUMENT, "%s: NULL pointer", name);
    if (((uintptr_t)b.ptr) % align != 0)
        return fail(TA_ERR_INVALID_ARGUMENT, "%s: pointer must be %zu-byte aligned", name, align);
    if (b.bytes < need_bytes)
        return fail(TA_ERR_BUFFER_TOO_SMALL, "%s buffer too small: have %llu bytes, need >= %llu", name,
                    (unsigned long long)b.bytes, (unsigned long long)need_bytes);
    return TA_OK;
}

ta_status check_dtype(const ta_buf &b, const char *name, int want) {
    if (b.dtype != want)
        return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: %s dtype must be %s, got %s", name,
                    dtype_name(want), dtype_name(b.dtype));
    return TA_OK;
}

#define TA_TRY(x)                      \
    do {                               \
        ta_status _s = (x);            \
        if (_s != TA_OK) return _s;    \
    } while (0)

struct TreePlan {
    TreeArgs a;
    int kv_type;
    bool use_tc;
    void *k, *v;
};

// cuTensorMapEncodeTiled from the driver, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
    std::call_once(g_encode_once, [] {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else
            cudaGetLastError();
    });
    return g_encode != nullptr;
}

bool encode_map(CUtensorMap *m, bool bf16, void *ptr, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                const cuuint32_t *box) {
    const cuuint32_t es[3] = {1, 1, 1};
    return g_encode(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, rank, ptr, dims,
                    strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

ta_status plan_tree(const ta_tree_params *p, int kernel, const ta_buf *q, const ta_buf *k, const ta_buf *v,
                    const ta_buf *mask, const ta_buf *tmp, const ta_buf *out, int window_start,
                    TreePlan *plan, const ta_buf *parents = nullptr) {
    if (kernel < TA_KERNEL_AUTO || kernel > TA_KERNEL_TENSOR_CORES)
        return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: kernel must be 0 (auto), 1 or 2, got %d", kernel);
    TA_TRY(check_tree_params(p, mask != nullptr));
    if (parents) {
        TA_TRY(check_dtype(*parents, "parents", TA_I32));
        if (p->q_l > p->kv_seq_len)
            return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: q_l (%u) must be <= kv_seq_len (%u)", p->q_l,
                        p->kv_seq_len);
        if (p->q_l > (uint32_t)kMaxTreeBitsNodes)
            return fail(TA_ERR_UNSUPPORTED, "tree_attention: a parent-array mask takes q_l <= %d (got %u); "
                        "build a dense mask with tree_mask_build instead", kMaxTreeBitsNodes, p->q_l);
    }
    // dtype contract (tree_attention.rs validate_buffers; bf16 K/V added)
    TA_TRY(check_dtype(*q, "q", TA_F32));
    if (k->dtype != v->dtype)
        return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: k.dtype (%s) must match v.dtype (%s)",
                    dtype_name(k->dtype), dtype_name(v->dtype));
    if (k->dtype != TA_F32 && k->dtype != TA_F16 && k->dtype != TA_BF16)
        return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: k/v dtype must be F32, F16 or BF16, got %s",
                    dtype_name(k->dtype));
    if (mask) TA_TRY(check_dtype(*mask, "tree_mask", TA_F32));
    TA_TRY(check_dtype(*out, "output", TA_F32));
    TA_TRY(check_dtype(*tmp, "tmp", TA_F32));

    // byte-length contract, overflow-checked
    uint64_t req_q, req_kv, req_mask = 0;
    if (!mul4(p->n_heads, p->q_l, p->head_dim, 4, &req_q))
        return fail(TA_ERR_OVERFLOW, "tree_attention: num_heads*q_seq_len*head_dim*4 overflows");
    if (!mul4(p->n_kv_heads, p->kv_capacity, p->head_dim, elt_bytes(k->dtype), &req_kv))
        return fail(TA_ERR_OVERFLOW, "tree_attention: num_kv_heads*kv_capacity*head_dim overflows");
    if (mask && !mul3(p->q_l, p->mask_stride, 4, &req_mask))
        return fail(TA_ERR_OVERFLOW, "tree_attention: q_seq_len*mask_stride*4 overflows");
    const uint32_t nwg = resolve_tree_nwg(p);
    if (nwg == 0) return fail(TA_ERR_CUDA, "tree_attention: no CUDA device to size the split count for");
    TreeWorkspace ws;
    if (!tree_workspace(p, nwg, &ws)) return fail(TA_ERR_OVERFLOW, "tree_attention: workspace size overflows");

    TA_TRY(check_buf(*q, "tree_attention: q", req_q, 16));
    TA_TRY(check_buf(*k, "tree_attention: k", req_kv, 16));
    TA_TRY(check_buf(*v, "tree_attention: v", req_kv, 16));
    if (mask) TA_TRY(check_buf(*mask, "tree_attention: tree_mask", req_mask, 4));
    if (parents) TA_TRY(check_buf(*parents, "tree_attention: parents", (uint64_t)p->q_l * 4u, 4));
    TA_TRY(check_buf(*out, "tree_attention: output", req_q, 16));
    TA_TRY(check_buf(*tmp, "tree_attention: tmp", ws.total, 16));

    TreeArgs &a = plan->a;
    a = TreeArgs{};
    a.q = static_cast<const float *>(q->ptr);
    a.k = k->ptr;
    a.v = v->ptr;
    a.mask = mask ? static_cast<const float *>(mask->ptr) : nullptr;
    char *t = static_cast<char *>(tmp->ptr);
    if (parents) {
        a.parents = static_cast<const int32_t *>(parents->ptr);
        a.anc = reinterpret_cast<const uint32_t *>(t + ws.off_anc);
        a.anc_words = (int)((p->q_l + 31u) / 32u);
    }
    a.part_o = reinterpret_cast<float *>(t + ws.off_part_o);
    a.part_ml = reinterpret_cast<float *>(t + ws.off_part_ml);
    a.cls = reinterpret_cast<uint8_t *>(t + ws.off_cls);
    a.q16 = t + ws.off_q16;
    a.err = reinterpret_cast<int *>(t + ws.off_err);
    a.out = static_cast<float *>(out->ptr);
    a.H = (int)p->n_heads;
    a.Hk = (int)p->n_kv_heads;
    a.D = (int)p->head_dim;
    a.N = (int)p->kv_seq_len;
    a.C = (int)p->kv_capacity;
    a.L = (int)p->q_l;
    a.stride = (int)p->mask_stride;
    a.nwg = (int)nwg;
    a.g = a.H / a.Hk;
    a.R = a.g * a.L;
    a.n_chunks = (a.N + 31) / 32;
    a.window_start = window_start;
    a.scale = p->scale;
    plan->kv_type = k->dtype == TA_F32 ? kKvF32 : (k->dtype == TA_F16 ? kKvF16 : kKvBF16);
    plan->k = k->ptr;
    plan->v = v->ptr;
    // Tensor cores when the K/V type is 16-bit and a KV head serves >= 16 query
    // rows (a dense contraction); otherwise the CUDA-core kernel.
    plan->use_tc = kernel != TA_KERNEL_CUDA_CORES && plan->kv_type != kKvF32 && a.R >= 16;
    a.q16_type = plan->use_tc ? plan->kv_type : -1;
    // partial slots left for the merge pass (0 = the main pass writes the output)
    a.cluster_x = 1;
    a.flat_groups = plan->use_tc ? tree_flat_groups(p) : 0;
    if (plan->use_tc) {
        int cx, cy;
        tree_tc_cluster_shape(a, &cx, &cy);
        a.cluster_x = cx;
    }
    a.n_part = a.nwg / a.cluster_x == 1 ? 0 : a.nwg / a.cluster_x;
    if (plan->use_tc && tree_tc_pairs(a.R, a.D) && (uint64_t)a.nwg * 2u > 65535u)
        return fail(TA_ERR_UNSUPPORTED, "tree_attention: nwg (%d) too large for the tensor-core kernel's grid", a.nwg);
    if (plan->use_tc && !get_encoder())
        return fail(TA_ERR_CUDA, "tree_attention: cuTensorMapEncodeTiled is not available");
    return TA_OK;
}

ta_status run_tree(const TreePlan &plan, cudaStream_t s) {
    TcMaps maps;
    if (plan.use_tc) {
        const TreeArgs &a = plan.a;
        const bool bf16 = plan.kv_type == kKvBF16;
        const cuuint64_t qdims[2] = {(cuuint64_t)a.D, (cuuint64_t)a.H * a.L};
        const cuuint64_t qstr[1] = {(cuuint64_t)a.D * 2};
        const cuuint32_t qbox[2] = {64, 128};
        const cuuint64_t kdims[3] = {(cuuint64_t)a.D, (cuuint64_t)a.N, (cuuint64_t)a.Hk};
        const cuuint64_t kstr[2] = {(cuuint64_t)a.D * 2, (cuuint64_t)a.C * a.D * 2};
        const cuuint32_t kbox[3] = {64, 32, 1}, kbox64[3] = {64, 64, 1};
        if (!encode_map(&maps.q16, bf16, a.q16, 2, qdims, qstr, qbox) ||
            !encode_map(&maps.k, bf16, plan.k, 3, kdims, kstr, kbox) ||
            !encode_map(&maps.v, bf16, plan.v, 3, kdims, kstr, kbox) ||
            !encode_map(&maps.k64, bf16, plan.k, 3, kdims, kstr, kbox64) ||
            !encode_map(&maps.v64, bf16, plan.v, 3, kdims, kstr, kbox64))
            return fail(TA_ERR_CUDA, "tree_attention: TMA descriptor encoding failed");
    }
    cudaError_t e = launch_tree_classify(plan.a, s);
    if (e != cudaSuccess) return cuda_fail(e, "tree_attention: chunk classification launch");
    e = plan.use_tc ? launch_tree_tc(plan.a, maps, plan.kv_type, s) : launch_tree_fma(plan.a, plan.kv_type, s);
    if (e != cudaSuccess) return cuda_fail(e, "tree_attention: main pass launch");
    return TA_OK;
}

// --------------------------------------------------------------- quant params
ta_status check_quant_params(const ta_quant_params *p) {
    if (p == nullptr) return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa: params is NULL");
    if (p->batch == 0 || p->n_q_heads == 0 || p->n_kv_heads == 0)
        return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa: batch, n_q_heads and n_kv_heads must be > 0");
    if (p->n_q_heads % p->n_kv_heads != 0)
        return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa: n_q_heads (%u) must be divisible by n_kv_heads (%u)",
                    p->n_q_heads, p->n_kv_heads);
    if (p->bits != 4 && p->bits != 8)
        return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa: bits must be 4 or 8, got %u", p->bits);
    const uint32_t pf = 32 / p->bits;
    if (p->dim == 0 || p->dim % pf != 0)
        return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa: dim (%u) must be a positive multiple of 32/bits (%u)",
                    p->dim, pf);
    if (p->group_size == 0 || p->dim % p->group_size != 0)
        return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa: dim (%u) must be a multiple of group_size (%u)", p->dim,
                    p->group_size);
    if (p->tokens == 0) return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa: tokens must be > 0");
    if (p->has_sinks > 1) return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa: has_sinks must be 0 or 1");
    if (p->kernel > (uint32_t)TA_KERNEL_WARP_MMA)
        return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa: kernel must be 0 (auto), 1, 2 or 3, got %u", p->kernel);
    if (!std::isfinite(p->scale)) return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa: scale is not finite");
    if (p->group_size % (4 * pf) != 0)
        return fail(TA_ERR_UNSUPPORTED,
                    "quant_sdpa: group_size must be a multiple of 4 * 32/bits (whole 16-byte word groups)");
    if (p->dim > 512) return fail(TA_ERR_UNSUPPORTED, "quant_sdpa: dim > 512 is not implemented");
    const uint64_t rows = (uint64_t)p->batch * p->n_q_heads;
    const uint64_t kvr = (uint64_t)p->batch * p->n_kv_heads;
    uint64_t cells;
    if (!mul3(kvr, p->tokens, p->dim, &cells) || rows > (uint64_t)INT_MAX || kvr > 65535u ||
        p->tokens > (uint32_t)INT_MAX)
        return fail(TA_ERR_UNSUPPORTED, "quant_sdpa: sizes exceed the kernels' index range");
    return TA_OK;
}

uint32_t window_tokens(const ta_quant_params *p) {
    return p->window_size == 0 ? p->tokens : (p->window_size < p->tokens ? p->window_size : p->tokens);
}

// Chunks of one KV row inside the window (chunks start at multiples of the
// kernel instance's chunk length).
uint32_t quant_chunks(const ta_quant_params *p) {
    const uint32_t t_lo = p->tokens - window_tokens(p);
    const uint32_t c = (uint32_t)quant_chunk_tokens((int)p->dim, (int)p->bits);
    return (p->tokens + c - 1u) / c - t_lo / c;
}

int quant_fallback_family(const ta_quant_params *p);

// Row groups per KV row of the CUDA-core or warp-MMA kernel (whichever the
// call runs when the tcgen05 kernel does not take it).
uint32_t quant_row_groups(const ta_quant_params *p) {
    const uint32_t rep = p->n_q_heads / p->n_kv_heads;
    const uint32_t rows = quant_fallback_family(p) == TA_KERNEL_WARP_MMA
                              ? (uint32_t)quant_mma_rows((int)rep, (int)p->dim, (int)p->group_size)
                              : (uint32_t)kQuantRowsPerCta;
    return (rep + rows - 1) / rows;
}

// Tensor-core quantized kernel: shape rules (params only, so that the split
// count and tmp size do not depend on which masks a call passes): head
// dimension 64, 128 or 256; TMEM for O (dim columns) and two score buffers
// (groups x rows per CTA each) within 512 columns; the worst-case shared-memory
// layout (both masks, shallowest rings) within the per-CTA limit.
struct QtcShape {
    int rr, rp, n_rb, cols;   // rows per CTA, MMA N (max(16, rr)), row blocks, TMEM columns
};
bool quant_tc_shape(const ta_quant_params *p, QtcShape *sh) {
    const int path = (int)p->kernel;
    if (path == TA_KERNEL_CUDA_CORES || path == TA_KERNEL_WARP_MMA) return false;
    if (p->dim != 64 && p->dim != 128 && p->dim != 256) return false;
    const int rep = (int)(p->n_q_heads / p->n_kv_heads);
    // automatic choice: the tensor-core kernel from 16 query rows per KV row
    // (draft-tree verification), where the CUDA-core kernel's per-row work
    // dominates, unless the warp-MMA kernel's wide form (16 rows per warp) takes
    // the shape: it measured faster there (4-bit draft tree of 256 rows on 8 KV
    // heads, dim 128: 29.4 against 41.4 us; 8-bit: 35.0 against 49.7)
    if (path == TA_KERNEL_AUTO && rep < kQuantTcMinRows) return false;
    if (path == TA_KERNEL_AUTO && quant_mma_wide(rep, (int)p->dim, (int)p->group_size)) return false;
    const int ng = (int)(p->dim / p->group_size);
    const int wpt = (int)(p->dim * p->bits / 32);
    if (wpt % 4 != 0 || p->group_size % 16 != 0) return false;
    sh->rr = rep <= 4 ? 4 : rep <= 8 ? 8 : rep <= 16 ? 16 : 32;
    sh->rp = sh->rr < 16 ? 16 : sh->rr;
    sh->n_rb = (rep + sh->rr - 1) / sh->rr;
    // TMEM: O^T (dimensions on lanes) takes rows-per-CTA columns per 128
    // dimensions, then the two score buffers
    const int ob = p->dim >= 128 ? (int)p->dim / 128 : 1;
    const int need = ob * sh->rp + 2 * ng * sh->rp;
    if (need > 512) return false;
    int cols = 32;
    while (cols < need) cols <<= 1;
    sh->cols = cols;
    const QtcLayout L = qtc_layout(sh->rp, (int)p->dim, wpt, ng, 4, 2, 2, true, true);
    return (size_t)L.total <= kQuantMaxSmem;
}

// Ring depths for the masks a call passes: the decoded K and V rings hold two
// tile parts (dim / 64 chunks each) each where shared memory allows, else one,
// else two chunks; the packed-K / packed-V rings three or two tiles; the
// deepest combination that fits.  The size is padded so that one CTA runs per
// SM (the TMEM budget assumes it).
struct QtcPlan {
    int nd, nk, nv;
    size_t smem;
};
bool quant_tc_plan(const ta_quant_params *p, const QtcShape &sh, bool has_mb, bool has_mf, QtcPlan *pl) {
    const int ng = (int)(p->dim / p->group_size);
    const int wpt = (int)(p->dim * p->bits / 32);
    const int nch = (int)p->dim / 64;
    // decoded chunks per ring (K and V each): two tile parts, one, or two chunks
    const int per_ring[3] = {2 * nch, nch, 2};
    for (int i = 0; i < 3; ++i)
        for (int n = 3; n >= 2; --n) {
            if (i > 0 && per_ring[i] >= per_ring[i - 1]) continue;
            const int nd = 2 * per_ring[i];
            if (nd > kQuantTcMaxRing) continue;
            const QtcLayout L = qtc_layout(sh.rp, (int)p->dim, wpt, ng, nd, n, n, has_mb, has_mf);
            if ((size_t)L.total > kQuantMaxSmem) continue;
            pl->nd = nd;
            pl->nk = pl->nv = n;
            pl->smem = (size_t)L.total < 120 * 1024 ? 120 * 1024 : (size_t)L.total;
            return true;
        }
    return false;
}

// Kernel of a quantized call when the tcgen05 kernel does not take it: the
// warp-MMA kernel where its shape rules allow (automatic choice or forced),
// else the CUDA-core kernel.
int quant_fallback_family(const ta_quant_params *p) {
    const int path = (int)p->kernel;
    if ((path == TA_KERNEL_AUTO || path == TA_KERNEL_WARP_MMA) &&
        quant_mma_shape_ok((int)p->dim, (int)p->group_size))
        return TA_KERNEL_WARP_MMA;
    return TA_KERNEL_CUDA_CORES;
}

int quant_family(const ta_quant_params *p) {
    QtcShape sh;
    return quant_tc_shape(p, &sh) ? (int)TA_KERNEL_TENSOR_CORES : quant_fallback_family(p);
}

uint32_t window_tiles(const ta_quant_params *p, uint32_t *j_lo) {
    const uint32_t t_lo = p->tokens - window_tokens(p);
    *j_lo = t_lo / 128u;
    return (p->tokens + 127u) / 128u - *j_lo;
}

// Token splits: as many as fill every SM's resident one-warp CTAs in one wave
// (kv rows x row groups x splits), at most one per chunk; for the tensor-core
// kernel, one CTA per SM over (kv rows x row blocks x splits), at most one
// split per 128-token tile.
uint32_t resolve_quant_nwg(const ta_quant_params *p) {
    if (p->nwg != 0) return p->nwg;
    const int sms = sm_count();
    if (sms <= 0) return 0;
    QtcShape sh;
    if (quant_tc_shape(p, &sh)) {
        const uint64_t units = (uint64_t)p->batch * p->n_kv_heads * (uint64_t)sh.n_rb;
        uint64_t nwg = (uint64_t)sms / units;
        uint32_t j_lo;
        const uint64_t nt = window_tiles(p, &j_lo);
        if (nwg > nt) nwg = nt;
        if (nwg < 1) nwg = 1;
        if (nwg > 65535) nwg = 65535;
        return (uint32_t)nwg;
    }
    const int ng = (int)(p->dim / p->group_size);
    const int per_sm = quant_fallback_family(p) == TA_KERNEL_WARP_MMA
                           ? quant_mma_ctas_per_sm((int)p->bits, (int)p->dim, ng,
                                                   (int)(p->n_q_heads / p->n_kv_heads))
                           : quant_ctas_per_sm((int)p->bits, (int)p->dim, ng);
    if (per_sm <= 0) return 0;
    const uint64_t units = (uint64_t)p->batch * p->n_kv_heads * quant_row_groups(p);
    uint64_t nwg = ((uint64_t)sms * (uint64_t)per_sm) / units;
    const uint64_t nch = quant_chunks(p);
    if (nwg > nch) nwg = nch;
    if (nwg < 1) nwg = 1;
    if (nwg > 65535) nwg = 65535;
    return (uint32_t)nwg;
}

// tmp = [error word region][split partials O (f32) then (S, M) pairs].
bool quant_tmp(const ta_quant_params *p, uint32_t nwg, uint64_t *bytes) {
    if (nwg <= 1) { *bytes = kQuantErrBytes; return true; }
    const uint64_t rows = (uint64_t)p->batch * p->n_q_heads;
    uint64_t part;
    if (!mul4(rows, nwg, (uint64_t)p->dim + 2, 4, &part)) return false;
    *bytes = part + kQuantErrBytes;
    return true;
}

}  // namespace

void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

void set_last_error(const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
}

}  // namespace ta

using namespace ta;

// ============================================================== exported ABI
TA_EXPORT size_t tree_attn_tmp_bytes(uint32_t n_heads, uint32_t head_dim, uint32_t q_l, uint32_t nwg) {
    const uint64_t nrows = sat_mul(n_heads, q_l);
    const uint64_t dv2 = (uint64_t)head_dim + 2;
    const uint64_t r = sat_mul(sat_mul(sat_mul(nrows, nwg), dv2), sizeof(float));
    return r > SIZE_MAX ? SIZE_MAX : (size_t)r;
}

TA_EXPORT uint32_t tree_attn_num_splits(const ta_tree_params *p) {
    if (check_tree_params(p, false) != TA_OK) return 0;
    return resolve_tree_nwg(p);
}

TA_EXPORT size_t tree_attn_workspace_bytes(const ta_tree_params *p) {
    if (check_tree_params(p, false) != TA_OK) return SIZE_MAX;
    const uint32_t nwg = resolve_tree_nwg(p);
    if (nwg == 0) return SIZE_MAX;
    TreeWorkspace ws;
    if (!tree_workspace(p, nwg, &ws)) return SIZE_MAX;
    return ws.total;
}

TA_EXPORT ta_status tree_attn_fwd_ex(const ta_tree_params *p, const ta_tree_options *o, const ta_buf *q,
                                     const ta_buf *k, const ta_buf *v, const ta_buf *mask, const ta_buf *tmp,
                                     const ta_buf *out, void *stream) {
    if (o == nullptr) return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: options is NULL");
    if (o->reserved != 0) return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: options.reserved must be 0");
    TreePlan plan;
    switch (o->mask_kind) {
        case TA_MASK_DENSE:
            if (absent(mask)) return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: TA_MASK_DENSE needs a mask");
            TA_TRY(plan_tree(p, o->kernel, &deref(q), &deref(k), &deref(v), mask, &deref(tmp), &deref(out), 0,
                             &plan));
            break;
        case TA_MASK_CAUSAL:
            if (o->window_start > (uint32_t)INT_MAX)
                return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: window_start out of range");
            TA_TRY(plan_tree(p, o->kernel, &deref(q), &deref(k), &deref(v), nullptr, &deref(tmp), &deref(out),
                             (int)o->window_start, &plan));
            break;
        case TA_MASK_PARENTS:
            if (absent(mask)) return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: TA_MASK_PARENTS needs parents");
            TA_TRY(plan_tree(p, o->kernel, &deref(q), &deref(k), &deref(v), nullptr, &deref(tmp), &deref(out), 0,
                             &plan, mask));
            break;
        default:
            return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: unknown mask_kind %d", o->mask_kind);
    }
    return run_tree(plan, static_cast<cudaStream_t>(stream));
}

TA_EXPORT ta_status tree_attn_fwd(const ta_tree_params *p, const ta_buf *q, const ta_buf *k,
                                  const ta_buf *v, const ta_buf *mask, const ta_buf *tmp,
                                  const ta_buf *out, void *stream) {
    const ta_tree_options o = {TA_KERNEL_AUTO, absent(mask) ? TA_MASK_CAUSAL : TA_MASK_DENSE, 0, 0};
    return tree_attn_fwd_ex(p, &o, q, k, v, mask, tmp, out, stream);
}

TA_EXPORT ta_status tree_attn_fwd_causal(const ta_tree_params *p, uint32_t window_start, const ta_buf *q,
                                         const ta_buf *k, const ta_buf *v, const ta_buf *tmp,
                                         const ta_buf *out, void *stream) {
    const ta_tree_options o = {TA_KERNEL_AUTO, TA_MASK_CAUSAL, window_start, 0};
    return tree_attn_fwd_ex(p, &o, q, k, v, nullptr, tmp, out, stream);
}

TA_EXPORT ta_status tree_attn_fwd_parents(const ta_tree_params *p, const ta_buf *parents, const ta_buf *q,
                                          const ta_buf *k, const ta_buf *v, const ta_buf *tmp, const ta_buf *out,
                                          void *stream) {
    if (absent(parents)) return fail(TA_ERR_INVALID_ARGUMENT, "tree_attention: parents is NULL");
    const ta_tree_options o = {TA_KERNEL_AUTO, TA_MASK_PARENTS, 0, 0};
    return tree_attn_fwd_ex(p, &o, q, k, v, parents, tmp, out, stream);
}

TA_EXPORT size_t tree_attn_status_offset(const ta_tree_params *p) {
    if (check_tree_params(p, false) != TA_OK) return SIZE_MAX;
    const uint32_t nwg = resolve_tree_nwg(p);
    if (nwg == 0) return SIZE_MAX;
    TreeWorkspace ws;
    if (!tree_workspace(p, nwg, &ws)) return SIZE_MAX;
    return ws.off_err;
}

TA_EXPORT ta_status tree_attn_reduce(const ta_tree_params *p, const ta_buf *tmp_d, const ta_buf *out_d,
                                     void *stream) {
    const ta_buf &tmp = deref(tmp_d), &out = deref(out_d);
    TA_TRY(check_tree_params(p, false));
    TA_TRY(check_dtype(tmp, "tmp", TA_F32));
    TA_TRY(check_dtype(out, "output", TA_F32));
    const uint32_t nwg = resolve_tree_nwg(p);
    if (nwg == 0) return fail(TA_ERR_CUDA, "tree_attention: no CUDA device to size the split count for");
    TreeWorkspace ws;
    uint64_t req_out;
    if (!tree_workspace(p, nwg, &ws) || !mul4(p->n_heads, p->q_l, p->head_dim, 4, &req_out))
        return fail(TA_ERR_OVERFLOW, "tree_attention: size overflows");
    TA_TRY(check_buf(tmp, "tree_attention: tmp", ws.total, 16));
    TA_TRY(check_buf(out, "tree_attention: output", req_out, 16));
    if (nwg == 1) return TA_OK;   // the main pass already wrote the output
    TreeArgs a{};
    char *t = static_cast<char *>(tmp.ptr);
    a.part_o = reinterpret_cast<float *>(t + ws.off_part_o);
    a.part_ml = reinterpret_cast<float *>(t + ws.off_part_ml);
    a.err = reinterpret_cast<int *>(t + ws.off_err);   // [1]: partial count the main pass left
    a.out = static_cast<float *>(out.ptr);
    a.H = (int)p->n_heads;
    a.L = (int)p->q_l;
    a.D = (int)p->head_dim;
    a.nwg = (int)nwg;
    cudaError_t e = launch_tree_reduce(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tree_attention: reduce launch");
    return TA_OK;
}

TA_EXPORT ta_status tree_mask_build(const ta_tree_params *p, const ta_buf *parents_d, const ta_buf *mask_d,
                                    void *stream) {
    const ta_buf &parents = deref(parents_d), &mask = deref(mask_d);
    TA_TRY(check_tree_params(p, true));
    if (p->q_l > p->kv_seq_len)
        return fail(TA_ERR_INVALID_ARGUMENT, "tree_mask_build: q_l (%u) must be <= kv_seq_len (%u)", p->q_l,
                    p->kv_seq_len);
    if (p->q_l > (uint32_t)kMaxTreeMaskNodes)
        return fail(TA_ERR_UNSUPPORTED, "tree_mask_build: q_l > %d is not implemented", kMaxTreeMaskNodes);
    TA_TRY(check_dtype(parents, "parents", TA_I32));
    TA_TRY(check_dtype(mask, "mask", TA_F32));
    uint64_t req_mask;
    if (!mul3(p->q_l, p->mask_stride, 4, &req_mask)) return fail(TA_ERR_OVERFLOW, "tree_mask_build: size overflows");
    TA_TRY(check_buf(parents, "tree_mask_build: parents", (uint64_t)p->q_l * 4, 4));
    TA_TRY(check_buf(mask, "tree_mask_build: mask", req_mask, 4));
    cudaError_t e = launch_tree_mask(static_cast<const int32_t *>(parents.ptr), (int)p->q_l, (int)p->kv_seq_len,
                                     (int)p->mask_stride, static_cast<float *>(mask.ptr),
                                     static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tree_mask_build: launch");
    return TA_OK;
}

TA_EXPORT uint32_t quant_sdpa_num_splits(const ta_quant_params *p) {
    if (check_quant_params(p) != TA_OK) return 0;
    return resolve_quant_nwg(p);
}

TA_EXPORT size_t quant_sdpa_tmp_bytes(const ta_quant_params *p) {
    if (check_quant_params(p) != TA_OK) return SIZE_MAX;
    const uint32_t nwg = resolve_quant_nwg(p);
    if (nwg == 0) return SIZE_MAX;
    uint64_t b;
    if (!quant_tmp(p, nwg, &b)) return SIZE_MAX;
    return (size_t)b;
}

namespace {

// quant_sdpa_fwd; first_wait_polls bounds the first copy wait of every CTA of
// the CUDA-core kernel (the normal bound for a regular call), and a call with
// a shorter bound must take that kernel.
ta_status quant_fwd_impl(const ta_quant_params *p, const ta_buf *queries_d, const ta_buf *k_packed_d,
                         const ta_buf *k_scales_d, const ta_buf *k_biases_d, const ta_buf *v_packed_d,
                         const ta_buf *v_scales_d, const ta_buf *v_biases_d, const ta_buf *sinks_d,
                         const ta_buf *mask_bool_d, const ta_buf *mask_float_d, const ta_buf *tmp_d,
                         const ta_buf *out_d, void *stream, uint32_t first_wait_polls, bool test_hook,
                         uint32_t tree_ql = 0, const ta_buf *parents_d = nullptr) {
    const ta_buf &queries = deref(queries_d), &k_packed = deref(k_packed_d), &k_scales = deref(k_scales_d);
    const ta_buf &k_biases = deref(k_biases_d), &v_packed = deref(v_packed_d), &v_scales = deref(v_scales_d);
    const ta_buf &v_biases = deref(v_biases_d), &sinks = deref(sinks_d), &mask_bool = deref(mask_bool_d);
    const ta_buf &mask_float = deref(mask_float_d), &tmp = deref(tmp_d), &out = deref(out_d);
    TA_TRY(check_quant_params(p));
    const int T = queries.dtype;
    if (T != TA_F16 && T != TA_BF16)
        return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa: queries dtype must be F16 or BF16, got %s",
                    dtype_name(T));
    const ta_buf *same_t[] = {&k_scales, &k_biases, &v_scales, &v_biases};
    const char *same_t_names[] = {"k_scales", "k_biases", "v_scales", "v_biases"};
    for (int i = 0; i < 4; ++i)
        if (same_t[i]->dtype != T)
            return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa: %s dtype must equal the queries dtype (%s), got %s",
                        same_t_names[i], dtype_name(T), dtype_name(same_t[i]->dtype));
    if (k_packed.dtype != TA_U32 || v_packed.dtype != TA_U32)
        return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa: k_packed and v_packed dtype must be U32");
    const bool has_bool = !absent(mask_bool_d);
    const bool has_float = !absent(mask_float_d);
    if (has_bool && mask_bool.dtype != TA_U32)
        return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa: mask_bool dtype must be U32");
    if (has_float && mask_float.dtype != T)
        return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa: mask_float dtype must equal the queries dtype");
    if (out.dtype != T && out.dtype != TA_F32)
        return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa: out dtype must be the queries dtype or F32");
    if (p->has_sinks && sinks.dtype != TA_F32)
        return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa: sinks dtype must be F32");

    const uint64_t rows = (uint64_t)p->batch * p->n_q_heads;
    const uint64_t kvr = (uint64_t)p->batch * p->n_kv_heads;
    const uint64_t words = p->dim / (32 / p->bits);
    const uint64_t groups = p->dim / p->group_size;
    uint64_t req_q, req_packed, req_sb, req_mb = 0, req_mf = 0, req_out, req_tmp;
    if (!mul3(rows, p->dim, 2, &req_q) || !mul4(kvr, p->tokens, words, 4, &req_packed) ||
        !mul4(kvr, p->tokens, groups, 2, &req_sb) || !mul3(rows, p->tokens, 4, &req_mb) ||
        !mul3(rows, p->tokens, 2, &req_mf) || !mul3(rows, p->dim, elt_bytes(out.dtype), &req_out))
        return fail(TA_ERR_OVERFLOW, "quant_sdpa: buffer size overflows");
    const uint32_t nwg = resolve_quant_nwg(p);
    if (nwg == 0) return fail(TA_ERR_CUDA, "quant_sdpa: no CUDA device to size the split count for");
    if (!quant_tmp(p, nwg, &req_tmp)) return fail(TA_ERR_OVERFLOW, "quant_sdpa: tmp size overflows");

    TA_TRY(check_buf(queries, "quant_sdpa: queries", req_q, 2));
    TA_TRY(check_buf(k_packed, "quant_sdpa: k_packed", req_packed, 16));
    TA_TRY(check_buf(v_packed, "quant_sdpa: v_packed", req_packed, 16));
    TA_TRY(check_buf(k_scales, "quant_sdpa: k_scales", req_sb, 2));
    TA_TRY(check_buf(k_biases, "quant_sdpa: k_biases", req_sb, 2));
    TA_TRY(check_buf(v_scales, "quant_sdpa: v_scales", req_sb, 2));
    TA_TRY(check_buf(v_biases, "quant_sdpa: v_biases", req_sb, 2));
    if (p->has_sinks) TA_TRY(check_buf(sinks, "quant_sdpa: sinks", (uint64_t)p->n_q_heads * 4, 4));
    if (tree_ql > 0) {
        // a draft tree over the last tree_ql tokens, as a parent array
        if (tree_ql > (uint32_t)kMaxQuantTreeNodes)
            return fail(TA_ERR_UNSUPPORTED, "quant_sdpa_fwd_tree: q_l (%u) must be <= %d", tree_ql, kMaxQuantTreeNodes);
        if (tree_ql > p->tokens)
            return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa_fwd_tree: q_l (%u) must be <= tokens (%u)", tree_ql,
                        p->tokens);
        if (p->n_q_heads % tree_ql != 0)
            return fail(TA_ERR_INVALID_ARGUMENT,
                        "quant_sdpa_fwd_tree: n_q_heads (%u) must be a multiple of q_l (%u): rows are (head, node)",
                        p->n_q_heads, tree_ql);
        if (absent(parents_d)) return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa_fwd_tree: parents is NULL");
        if (parents_d->dtype != TA_I32) return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa_fwd_tree: parents dtype must be I32");
        TA_TRY(check_buf(*parents_d, "quant_sdpa_fwd_tree: parents", (uint64_t)tree_ql * 4, 4));
    }
    if (has_bool) TA_TRY(check_buf(mask_bool, "quant_sdpa: mask_bool", req_mb, 4));
    if (has_float) TA_TRY(check_buf(mask_float, "quant_sdpa: mask_float", req_mf, 2));
    TA_TRY(check_buf(out, "quant_sdpa: out", req_out, out.dtype == TA_F32 ? 4 : 2));
    TA_TRY(check_dtype(tmp, "tmp", TA_F32));
    TA_TRY(check_buf(tmp, "quant_sdpa: tmp", req_tmp, 16));

    QuantArgs a{};
    a.queries = queries.ptr;
    a.kp = static_cast<const uint32_t *>(k_packed.ptr);
    a.vp = static_cast<const uint32_t *>(v_packed.ptr);
    a.ks = k_scales.ptr;
    a.kb = k_biases.ptr;
    a.vs = v_scales.ptr;
    a.vb = v_biases.ptr;
    a.sinks = p->has_sinks ? static_cast<const float *>(sinks.ptr) : nullptr;
    a.mbool = has_bool ? static_cast<const uint32_t *>(mask_bool.ptr) : nullptr;
    a.mfloat = has_float ? mask_float.ptr : nullptr;
    a.err = static_cast<int *>(tmp.ptr);
    if (nwg > 1) {
        a.part_o = reinterpret_cast<float *>(static_cast<unsigned char *>(tmp.ptr) + kQuantErrBytes);
        a.part_ml = a.part_o + rows * nwg * p->dim;
    }
    a.out = out.ptr;
    a.rows = (int)rows;
    a.nQ = (int)p->n_q_heads;
    a.rep = (int)(p->n_q_heads / p->n_kv_heads);
    a.kv_rows = (int)kvr;
    a.dim = (int)p->dim;
    a.N = (int)p->tokens;
    a.bits = (int)p->bits;
    a.G = (int)p->group_size;
    a.has_sinks = (int)p->has_sinks;
    a.window = (int)p->window_size;
    a.nwg = (int)nwg;
    a.wpt = (int)(p->dim * p->bits / 32);
    a.ng = (int)(p->dim / p->group_size);
    a.n_rg = (int)quant_row_groups(p);
    a.t_lo = (int)(p->tokens - window_tokens(p));
    a.c_lo = a.t_lo / quant_chunk_tokens(a.dim, a.bits);
    a.nch = (int)quant_chunks(p);
    const auto al16 = [](const void *ptr) { return ((uintptr_t)ptr & 15u) == 0; };
    a.al_sb = al16(k_scales.ptr) && al16(k_biases.ptr) && al16(v_scales.ptr) && al16(v_biases.ptr) &&
              ((uint64_t)p->tokens * a.ng * 2) % 16 == 0;
    a.al_mb = has_bool && al16(mask_bool.ptr) && p->tokens % 4 == 0;
    a.al_mf = has_float && al16(mask_float.ptr) && p->tokens % 8 == 0;
    if ((uint64_t)a.nwg * a.n_rg > (uint64_t)INT_MAX)
        return fail(TA_ERR_UNSUPPORTED, "quant_sdpa: too many splits x row groups");
    a.t_is_bf16 = T == TA_BF16;
    a.out_f32 = out.dtype == TA_F32;
    a.scale = p->scale;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    QtcShape sh;
    QtcPlan pl;
    a.first_wait_polls = first_wait_polls;
    a.tree_ql = (int)tree_ql;
    a.tree_parents = tree_ql > 0 ? static_cast<const int32_t *>(parents_d->ptr) : nullptr;
    const bool use_tc = quant_tc_shape(p, &sh) && quant_tc_plan(p, sh, has_bool, has_float, &pl);
    if (test_hook && use_tc)
        return fail(TA_ERR_UNSUPPORTED, "quant_sdpa: the wait-limit test hook takes the CUDA-core or warp-MMA "
                    "kernel only (set kernel = 1 or 3)");
    if (use_tc) {
        uint32_t j_lo;
        a.ntile = (int)window_tiles(p, &j_lo);
        a.j_lo = (int)j_lo;
        a.rp = sh.rr;
        a.n_rb = sh.n_rb;
        a.tc_cols = sh.cols;
        a.tc_nd = pl.nd;
        a.tc_nk = pl.nk;
        a.tc_nv = pl.nv;
        if ((uint64_t)kvr * (uint64_t)sh.n_rb > 65535u)
            return fail(TA_ERR_UNSUPPORTED, "quant_sdpa: too many KV rows x row blocks for one launch");
        e = launch_quant_tc(a, pl.smem, s);
    } else if (quant_fallback_family(p) == TA_KERNEL_WARP_MMA) {
        e = launch_quant_mma(a, s);
    } else {
        e = launch_quant_fma(a, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "quant_sdpa: main pass launch");
    if (nwg > 1) {
        e = launch_quant_merge(a, s);
        if (e != cudaSuccess) return cuda_fail(e, "quant_sdpa: merge launch");
    }
    return TA_OK;
}

}  // namespace

TA_EXPORT ta_status quant_sdpa_fwd(const ta_quant_params *p, const ta_buf *queries, const ta_buf *k_packed,
                                   const ta_buf *k_scales, const ta_buf *k_biases, const ta_buf *v_packed,
                                   const ta_buf *v_scales, const ta_buf *v_biases, const ta_buf *sinks,
                                   const ta_buf *mask_bool, const ta_buf *mask_float, const ta_buf *tmp,
                                   const ta_buf *out, void *stream) {
    return quant_fwd_impl(p, queries, k_packed, k_scales, k_biases, v_packed, v_scales, v_biases, sinks, mask_bool,
                          mask_float, tmp, out, stream, kQuantWaitPolls, false);
}

TA_EXPORT ta_status quant_sdpa_fwd_tree(const ta_quant_params *p, uint32_t q_l, const ta_buf *parents,
                                        const ta_buf *queries, const ta_buf *k_packed, const ta_buf *k_scales,
                                        const ta_buf *k_biases, const ta_buf *v_packed, const ta_buf *v_scales,
                                        const ta_buf *v_biases, const ta_buf *sinks, const ta_buf *mask_bool,
                                        const ta_buf *tmp, const ta_buf *out, void *stream) {
    if (q_l == 0) return fail(TA_ERR_INVALID_ARGUMENT, "quant_sdpa_fwd_tree: q_l must be > 0");
    return quant_fwd_impl(p, queries, k_packed, k_scales, k_biases, v_packed, v_scales, v_biases, sinks, mask_bool,
                          nullptr, tmp, out, stream, kQuantWaitPolls, false, q_l, parents);
}

TA_EXPORT ta_status ta_test_quant_sdpa_fwd_wait_limit(uint32_t first_wait_polls, const ta_quant_params *p,
                                                      const ta_buf *queries, const ta_buf *k_packed,
                                                      const ta_buf *k_scales, const ta_buf *k_biases,
                                                      const ta_buf *v_packed, const ta_buf *v_scales,
                                                      const ta_buf *v_biases, const ta_buf *sinks,
                                                      const ta_buf *mask_bool, const ta_buf *mask_float,
                                                      const ta_buf *tmp, const ta_buf *out, void *stream) {
    return quant_fwd_impl(p, queries, k_packed, k_scales, k_biases, v_packed, v_scales, v_biases, sinks, mask_bool,
                          mask_float, tmp, out, stream, first_wait_polls, true);
}

TA_EXPORT const char *ta_last_error(void) { return g_err.c_str(); }

TA_EXPORT uint64_t ta_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

TA_EXPORT int quant_sdpa_kernel_family(const ta_quant_params *p) {
    if (check_quant_params(p) != TA_OK) return -1;
    return quant_family(p);
}

TA_EXPORT int quant_sdpa_uses_tensor_cores(const ta_quant_params *p) {
    if (check_quant_params(p) != TA_OK) return -1;
    return quant_family(p) == TA_KERNEL_CUDA_CORES ? 0 : 1;
}
