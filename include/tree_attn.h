/*
 * tree_attn.h - C ABI of the GB300 (sm_103a) tree-verify attention library.
 *
 * The library computes the verification step of tree speculative decoding:
 * split-KV (flash-decoding) attention of q_l draft-tree queries per head over
 * a KV cache, with an explicit tree mask, GQA head mapping, an online softmax
 * (running max M and running sum S) per split and a second pass that merges
 * the per-split partials.  A second family attends over an affine-quantized
 * (4/8-bit packed) K/V cache with optional attention sinks, a sliding window,
 * a boolean and an additive float mask.
 *
 * Sources of the operations (web pages, by title and section):
 *   [TA-M]  mlx-native 0.9.1 src/shaders/tree_attention.metal - header comment
 *           (explicit mask, byte-identity contract), TreeAttentionParams struct,
 *           tree_attention_impl (chunk loop, mask early exit, QK, online softmax,
 *           PV, partial write).
 *   [TA-R]  mlx-native 0.9.2 src/mlx_native/ops/tree_attention.rs - validate_params,
 *           validate_buffers, tree_attention (buffer docs, two-pass dispatch),
 *           tmp_buffer_bytes, unit tests.
 *   [FQS]   metaltile-std 0.1.0 src/ffai/flash_quantized_sdpa.rs - module doc
 *           (layout, mask variants) and the three kernel macros.
 *
 * Conventions shared by every entry point:
 *   - Every buffer is borrowed device memory described by a ta_buf (pointer,
 *     usable byte count, element type) passed by address; the ta_buf itself
 *     is only read during the call.  An optional buffer is absent when its
 *     ta_buf pointer is NULL (or its `ptr` is NULL with `bytes` 0).
 *   - The library never allocates, frees, copies to the host or
 *     synchronizes; all work is enqueued on `stream` (a cudaStream_t passed
 *     as void*, NULL = legacy default stream).
 *   - All argument checks run before any launch, with overflow-checked size
 *     arithmetic.  On any non-TA_OK status nothing has been launched and no
 *     output was touched; ta_last_error() then returns a message for the
 *     calling thread.  TA_ERR_CUDA reports a failed launch (cudaGetLastError).
 *   - The functions are reentrant; concurrent calls must not share tmp buffers.
 */
#ifndef TREE_ATTN_H_
#define TREE_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TA_OK = 0,
    TA_ERR_INVALID_ARGUMENT = 1, /* bad shape, dtype, null pointer or alignment */
    TA_ERR_BUFFER_TOO_SMALL = 2, /* a ta_buf holds fewer bytes than the shapes need */
    TA_ERR_OVERFLOW = 3,         /* a size computation overflows 64 bits */
    TA_ERR_UNSUPPORTED = 4,      /* valid request the kernels do not implement */
    TA_ERR_CUDA = 5              /* the CUDA runtime reported an error */
} ta_status;

typedef enum { TA_F32 = 0, TA_F16 = 1, TA_BF16 = 2, TA_U32 = 3, TA_I32 = 4 } ta_dtype;

/*
 * Kernel family of a call (ta_tree_options.kernel, ta_quant_params.kernel).
 * TA_KERNEL_AUTO is the library's choice; the others force a family, for
 * tests and measurements.  The choice travels with the call: there is no
 * process-wide setting, so concurrent callers cannot affect one another.
 */
typedef enum {
    TA_KERNEL_AUTO = 0,         /* tensor cores where the shape makes a dense contraction */
    TA_KERNEL_CUDA_CORES = 1,   /* always the CUDA-core kernel */
    TA_KERNEL_TENSOR_CORES = 2, /* the tensor-core kernel wherever its shape rules allow it */
    TA_KERNEL_WARP_MMA = 3      /* quantized path only: the warp-MMA kernel wherever its
                                   shape rules allow it (the tree path rejects it) */
} ta_kernel;

/* Borrowed device buffer. `bytes` is the usable size starting at `ptr`. */
typedef struct {
    void *ptr;
    uint64_t bytes;
    int32_t dtype;    /* ta_dtype */
    int32_t reserved; /* must be 0 */
} ta_buf;

/*
 * Tree-attention parameters, 9 x 4 bytes = 36 bytes in the field order of the
 * GPU params struct ([TA-M] TreeAttentionParams; [TA-R] test_gpu_params_layout).
 *   n_heads      query heads H            n_kv_heads  KV heads Hk, H % Hk == 0
 *   head_dim     D in {128, 256, 512}     kv_seq_len  N valid KV positions, > 0
 *   kv_capacity  C >= N, stride (in rows) between KV heads
 *   scale        logit = (q . k) * scale + mask
 *   nwg          number of KV splits; 0 = library's choice (tree_attn_num_splits)
 *   q_l          L tree nodes (queries) per head, > 0
 *   mask_stride  floats between mask rows, >= N
 */
typedef struct {
    uint32_t n_heads;
    uint32_t n_kv_heads;
    uint32_t head_dim;
    uint32_t kv_seq_len;
    uint32_t kv_capacity;
    float scale;
    uint32_t nwg;
    uint32_t q_l;
    uint32_t mask_stride;
} ta_tree_params;

/*
 * Quantized-KV attention parameters ([FQS] module doc "Layout" and the
 * constexpr list of the kernels), as runtime values:
 *   batch B, n_q_heads nQ, n_kv_heads nKV (nQ % nKV == 0, repeat = nQ / nKV),
 *   dim (a multiple of 32/bits and of group_size), tokens N > 0, bits in {4, 8},
 *   group_size G, has_sinks in {0, 1}, window_size (0 = all tokens, else the
 *   last window_size tokens), scale (multiplies the query), nwg (splits, 0 = auto),
 *   kernel (ta_kernel; not from the pages).
 */
typedef struct {
    uint32_t batch;
    uint32_t n_q_heads;
    uint32_t n_kv_heads;
    uint32_t dim;
    uint32_t tokens;
    uint32_t bits;
    uint32_t group_size;
    uint32_t has_sinks;
    uint32_t window_size;
    float scale;
    uint32_t nwg;
    uint32_t kernel;   /* ta_kernel; the split count and tmp size follow the family chosen */
} ta_quant_params;

/* Mask forms of tree_attn_fwd_ex. */
typedef enum {
    TA_MASK_DENSE = 0,    /* `mask` is the [q_l, mask_stride] f32 mask (tree_attn_fwd) */
    TA_MASK_CAUSAL = 1,   /* implicit causal / sliding window; `mask` unused (tree_attn_fwd_causal) */
    TA_MASK_PARENTS = 2   /* `mask` is the [q_l] i32 parent array (tree_attn_fwd_parents) */
} ta_mask_kind;

/* Per-call options of tree_attn_fwd_ex (the pages' 36-byte params struct
 * stays as it is). */
typedef struct {
    int32_t kernel;         /* ta_kernel */
    int32_t mask_kind;      /* ta_mask_kind */
    uint32_t window_start;  /* TA_MASK_CAUSAL: first attended position */
    int32_t reserved;       /* must be 0 */
} ta_tree_options;

/* ------------------------------------------------------------------ tree */

/*
 * Bytes of the per-split partial results for n_heads * q_l rows and nwg
 * splits: rows * nwg * (head_dim + 2) * 4, saturating at SIZE_MAX
 * ([TA-R] tmp_buffer_bytes; 16 heads, D 256, q_l 1, NWG 32 -> 528384).
 */
size_t tree_attn_tmp_bytes(uint32_t n_heads, uint32_t head_dim, uint32_t q_l, uint32_t nwg);

/*
 * Number of KV splits (partial slots per output row) tree_attn_fwd will use
 * for these parameters on the current device: p->nwg when non-zero, else a
 * choice sized to the SM count.  With head dim 512, more than 128 rows per KV
 * head and p->nwg == 0 the tensor-core pass may spread the (KV head, key tile)
 * work of all heads evenly over every SM; a row's keys are then cut at
 * different points for different KV heads, and this count is the most slots
 * any row uses (slots a row does not use hold S = 0 and add nothing to the
 * merge).  Returns 0 when the parameters are invalid or no device is visible.
 */
uint32_t tree_attn_num_splits(const ta_tree_params *p);

/*
 * Bytes the `tmp` buffer of tree_attn_fwd / tree_attn_reduce must hold: the
 * partials (tree_attn_tmp_bytes at the resolved split count) plus a small
 * per-32-key-chunk classification area and a 16-bit copy of Q for the tensor
 * core path.  Returns SIZE_MAX on invalid parameters or overflow.
 */
size_t tree_attn_workspace_bytes(const ta_tree_params *p);

/*
 * Main pass ([TA-M] tree_attention_impl; [TA-R] tree_attention, first pass).
 *   q     [n_heads, q_l, head_dim] f32
 *   k, v  [n_kv_heads, kv_capacity, head_dim], same dtype, f32 / f16 / bf16;
 *         only positions [0, kv_seq_len) are read.
 *   mask  [q_l, mask_stride] f32, 0.0 = attend, -65504.0 = masked; cells at
 *         positions >= kv_seq_len are ignored.  The mask is added to the
 *         scaled logit.  A 32-key chunk whose cells are all <= -65504 for a
 *         row is skipped for that row; a chunk masked for every row is not
 *         loaded at all.  An absent mask selects the implicit causal mask
 *         (tree_attn_fwd_causal with window_start 0).
 *   tmp   f32, >= tree_attn_workspace_bytes(p) bytes, 16-byte aligned.
 *   out   [q_l, n_heads, head_dim] f32 (query-outer, head-inner: NOT Q's layout).
 * With one split the normalized output is written to `out` here and
 * tree_attn_reduce is a no-op; otherwise `out` is written by tree_attn_reduce.
 * A row that attends no key produces zeros.
 */
ta_status tree_attn_fwd(const ta_tree_params *p, const ta_buf *q, const ta_buf *k, const ta_buf *v,
                        const ta_buf *mask, const ta_buf *tmp, const ta_buf *out, void *stream);

/*
 * Main pass with the implicit causal / sliding-window mask of the parent
 * kernel ([TA-M] header comment): query row i attends positions
 * [window_start, kv_seq_len - q_l + i].  Same buffers as tree_attn_fwd minus
 * the mask.  For a mask buffer equal to this causal mask, tree_attn_fwd
 * produces a bit-identical output ([TA-M] byte-identity contract).
 */
ta_status tree_attn_fwd_causal(const ta_tree_params *p, uint32_t window_start, const ta_buf *q,
                               const ta_buf *k, const ta_buf *v, const ta_buf *tmp,
                               const ta_buf *out, void *stream);

/*
 * Main pass with the tree mask given compactly as a parent array instead of
 * a dense [q_l, mask_stride] f32 mask (the tree semantics of [TA-M]'s header
 * comment: node i of the draft tree sits at KV position kv_seq_len - q_l + i
 * and attends the prefix [0, kv_seq_len - q_l), its ancestors and itself).
 * The result is bit-identical to tree_attn_fwd given the mask
 * tree_mask_build writes for the same parents; no dense mask
 * is read or written (the mask-compaction pass builds a per-row ancestor
 * bitset of (q_l + 31) / 32 words in `tmp`; no extra launch).
 *   parents  [q_l] i32 on the device, the rule of tree_mask_build: a chain
 *            i, parents[i], ... ends at a value outside [0, current node).
 *   q, k, v, tmp, out  as for tree_attn_fwd; p->mask_stride is not used.
 * Errors: as tree_attn_fwd's checks; parents I32, >= 4*q_l bytes, 4-byte
 * aligned; q_l <= kv_seq_len; q_l > 256 is TA_ERR_UNSUPPORTED (use
 * tree_mask_build and tree_attn_fwd).  Nothing is launched on error.
 * tree_attn_reduce merges its partials as for tree_attn_fwd.
 */
ta_status tree_attn_fwd_parents(const ta_tree_params *p, const ta_buf *parents, const ta_buf *q,
                                const ta_buf *k, const ta_buf *v, const ta_buf *tmp, const ta_buf *out,
                                void *stream);

/*
 * The main pass of tree_attn_fwd, tree_attn_fwd_causal or tree_attn_fwd_parents
 * (chosen by o->mask_kind; `mask` is then the dense mask, unused, or the
 * parent array) with the kernel family of o->kernel.  Same buffers, checks,
 * workspace and results as those calls, which are this call with
 * TA_KERNEL_AUTO.  The workspace size and split count do not depend on the
 * family.  Errors: TA_ERR_INVALID_ARGUMENT for a NULL `o`, an unknown kernel
 * or mask kind, reserved != 0, or a missing mask / parent array.
 */
ta_status tree_attn_fwd_ex(const ta_tree_params *p, const ta_tree_options *o, const ta_buf *q,
                           const ta_buf *k, const ta_buf *v, const ta_buf *mask, const ta_buf *tmp,
                           const ta_buf *out, void *stream);

/*
 * Byte offset, inside the `tmp` buffer of the tree main pass, of the call's
 * 32-bit device status word (an int32).  The mask-compaction pass of every
 * main-pass call sets it to 0; the tensor-core main pass writes a non-zero
 * code there when one of its bounded waits (a K/V copy or an MMA that did not
 * complete within about two seconds) gave up, and the output of that call is
 * then not valid.  The library never reads it back: a caller that wants to
 * check copies the word to the host after the call (same stream) and tests it
 * for 0.  SIZE_MAX on invalid parameters.
 */
size_t tree_attn_status_offset(const ta_tree_params *p);

/*
 * Second pass ([TA-R] tree_attention, reduce pass): merges the nwg partials
 * of every (query, head) row with a log-sum-exp rescale:
 *   M* = max_w M_w,  S* = sum_w S_w e^(M_w - M*),
 *   out = sum_w O_w e^(M_w - M*) / S*   (0 when S* == 0);
 * a partial with S_w = 0 (no attended key) is skipped, its O_w not read.
 * `p` must equal the one given to the main pass; `tmp` is its tmp buffer.
 */
ta_status tree_attn_reduce(const ta_tree_params *p, const ta_buf *tmp, const ta_buf *out,
                           void *stream);

/*
 * The whole verify step (main pass and merge, same results as tree_attn_fwd
 * followed by tree_attn_reduce) for callers that cannot allocate device
 * memory: engines that plan every device byte up front, plugins inside a
 * framework that owns the allocator, decode loops that cannot afford the
 * synchronization an allocation may cause.  The pages have no counterpart;
 * this entry point exists for those callers only.
 *   Instead of a caller tmp buffer it uses one static device array of
 *   16 MiB (16777216 bytes) that every GPU loading the library holds until
 *   process exit.  Parameters whose tree_attn_workspace_bytes exceed that
 *   fail with TA_ERR_UNSUPPORTED (lower nwg, or use tree_attn_fwd).
 *   The array's device address is looked up on every call (it belongs to the
 *   CUDA context, which a cudaDeviceReset replaces); the first call in a
 *   context also loads the library's module there, so make that first call
 *   before any stream capture.
 *   It allocates nothing and calls no allocating routine.  All calls share the
 *   array and it keeps the last call's contents; nothing in it has to start
 *   at zero, but calls that overlap on the GPU race on it.
 * Buffers as for tree_attn_fwd (an absent mask = implicit causal mask).
 */
ta_status tree_attn_fwd_noalloc(const ta_tree_params *p, const ta_buf *q, const ta_buf *k,
                                const ta_buf *v, const ta_buf *mask, const ta_buf *out,
                                void *stream);

/*
 * Dense tree mask from a parent array, built on the device: the step before
 * the verify pass (the tree semantics of mlx-native tree_attention.metal's
 * header comment and of the tree_attention.rs tests; 0 = attend, -65504 =
 * masked).  The draft tree's node i sits at KV position kv_seq_len - q_l + i.
 *   p        q_l, kv_seq_len and mask_stride are used; p must pass the same
 *            checks as for tree_attn_fwd (mask_stride >= kv_seq_len >= q_l).
 *   parents  [q_l] i32 on the device: parents[i] in [-1, i) (node 0 is the
 *            root, -1 = no parent).  Node a is an ancestor of i when the chain
 *            i, parents[i], parents[parents[i]], ... reaches a; a value outside
 *            [0, current node) ends the chain there.
 *   mask     [q_l, mask_stride] f32 on the device, every cell written: row i is
 *            0 on [0, kv_seq_len - q_l), at kv_seq_len - q_l + a for i itself
 *            and each of its ancestors a, and -65504 elsewhere (including
 *            positions >= kv_seq_len).
 * Errors: as tree_attn_fwd's checks; parents must be I32 and 4-byte aligned,
 * mask F32 and 4-byte aligned; q_l > 16384 is TA_ERR_UNSUPPORTED.  Nothing is
 * launched on error.  Asynchronous on `stream`.
 */
ta_status tree_mask_build(const ta_tree_params *p, const ta_buf *parents, const ta_buf *mask, void *stream);

/* ----------------------------------------------------------------- quant */

/* Splits quant_sdpa_fwd will use (p->nwg when non-zero); 0 on invalid input. */
uint32_t quant_sdpa_num_splits(const ta_quant_params *p);

/* Bytes of the `tmp` buffer of quant_sdpa_fwd: 256 (error word region) plus,
 * with more than one split, B*nQ*nwg*(dim+2)*4 for the split partials;
 * SIZE_MAX on invalid parameters or overflow. */
size_t quant_sdpa_tmp_bytes(const ta_quant_params *p);

/*
 * Attention over an affine-quantized K/V cache ([FQS] all three kernel macros).
 *   queries   [B*nQ, dim] T (T = f16 or bf16), multiplied by `scale` once
 *   k_packed  [B*nKV, tokens, dim*bits/32] u32: element d of a token sits at
 *             bits (d % (32/bits)) * bits of word d / (32/bits)
 *   k_scales, k_biases  [B*nKV, tokens, dim/group_size] T:
 *             k[d] = scale[d / group_size] * code + bias[d / group_size]
 *   v_packed, v_scales, v_biases: same layout for V
 *   sinks     [nQ] f32, read when has_sinks: a virtual key with logit
 *             sinks[q % nQ] (not scaled) and value 0, counted once
 *   mask_bool [B*nQ, tokens] u32 or absent: 0 drops the token for that query
 *   mask_float[B*nQ, tokens] T or absent: added to the logit after the gates
 *   tmp       f32, >= quant_sdpa_tmp_bytes(p) bytes, 16-byte aligned.  Its
 *             first 32-bit word is an error word: the kernel ORs in 1 when a
 *             copy of K/V into shared memory did not complete within its
 *             wait bound (the output is then not valid).  The library never
 *             clears it; a caller that wants to check it zeroes it first.
 *   out       [B*nQ, dim], dtype T or f32; out = o / l when l > 0, else 0
 * Query q uses KV row q / (nQ / nKV).  Tokens outside the window are not read.
 * k_packed and v_packed must be 16-byte aligned.
 */
ta_status quant_sdpa_fwd(const ta_quant_params *p, const ta_buf *queries, const ta_buf *k_packed,
                         const ta_buf *k_scales, const ta_buf *k_biases, const ta_buf *v_packed,
                         const ta_buf *v_scales, const ta_buf *v_biases, const ta_buf *sinks,
                         const ta_buf *mask_bool, const ta_buf *mask_float, const ta_buf *tmp,
                         const ta_buf *out, void *stream);

/*
 * quant_sdpa_fwd for draft-tree verification on a quantized cache, with the
 * tree mask given as a parent array instead of a dense [B*nQ, tokens] float
 * mask (the tree semantics of [TA-M]'s header comment applied to the rows of
 * [FQS]): the q_l draft nodes are the last q_l tokens of the cache, query row
 * q is node q % q_l (rows ordered (batch, head, node), so n_q_heads counts
 * heads x q_l), and row q attends every token before the tree plus the tree
 * positions of its node's ancestors and of itself - the tokens an additive
 * float mask of 0 there and -65504 on the other tree positions leaves, with no
 * mask read from memory.  Window, bool mask and sinks apply as in
 * quant_sdpa_fwd; there is no float mask.
 *   q_l      1..32 nodes; n_q_heads must be a multiple of q_l; q_l <= tokens.
 *   parents  [q_l] i32 on the device, the rule of tree_mask_build (a chain i,
 *            parents[i], ... ends at a value outside [0, current node)).
 * Other buffers and errors as quant_sdpa_fwd; q_l > 32 is TA_ERR_UNSUPPORTED.
 */
ta_status quant_sdpa_fwd_tree(const ta_quant_params *p, uint32_t q_l, const ta_buf *parents,
                              const ta_buf *queries, const ta_buf *k_packed, const ta_buf *k_scales,
                              const ta_buf *k_biases, const ta_buf *v_packed, const ta_buf *v_scales,
                              const ta_buf *v_biases, const ta_buf *sinks, const ta_buf *mask_bool,
                              const ta_buf *tmp, const ta_buf *out, void *stream);

/* ----------------------------------------------------------------- misc */

/* Message for the calling thread's last non-TA_OK status ("" if none). */
const char *ta_last_error(void);

/* Kernels launched by this library in this process so far (host counter). */
uint64_t ta_launch_count(void);

/*
 * Kernel family quant_sdpa_fwd takes with these params (p->kernel included):
 * TA_KERNEL_TENSOR_CORES (the tcgen05 kernel), TA_KERNEL_WARP_MMA or
 * TA_KERNEL_CUDA_CORES; -1 for invalid params.  No device work.
 *
 * The warp-MMA kernel serves head dimensions 64, 128 and 256 with group size
 * 32 or 64, four query rows per CTA; from 16 query rows per KV row, with head
 * dimension 64 or 128, it runs 16 query rows per CTA instead (its wide form,
 * each score MMA within one scale group).  With TA_KERNEL_AUTO it is chosen
 * below 16 query rows per KV row, from 16 rows where the wide form takes the
 * shape, and wherever the tcgen05 kernel's rules fail: its
 * scores multiply the exact K codes with Q scaled per row by a power of two
 * into f16 (the group scales and biases are applied to the f32 sums), and P V
 * takes V dequantized once to f16 (s * code + b, one rounding) and P as two
 * f16 terms, as the tcgen05 kernel does; the same f16-range assumption on the
 * dequantized V values applies.
 */
int quant_sdpa_kernel_family(const ta_quant_params *p);

/*
 * 1 if quant_sdpa_fwd with these params (p->kernel included) takes a
 * tensor-core kernel (tcgen05 or warp MMA), 0 if the CUDA-core kernel, -1 for
 * invalid params.  No device work.
 *
 * The tensor-core kernel serves head dimensions 64, 128 and 256 when TMEM
 * holds O (dim f32 columns) and two score buffers (dim / group_size groups x
 * 16 or 32 query rows each) and its shared-memory layout fits.  With
 * TA_KERNEL_AUTO it is chosen from 16 query rows per KV row (e.g. draft-tree
 * nodes as rows) for the shapes the warp-MMA kernel's wide form does not take
 * (head dimension 256, group size other than 32 or 64).  It feeds the tensor core the exact integer codes of K (the
 * per-group scales and biases are applied to the f32 scores), V dequantized
 * once to f16 (s * code + b, one rounding) and the weights P as two f16 terms
 * (P_hi + P_lo); Q is scaled per row by a power of two into f16 (exact for
 * f16 and bf16 queries).  Dequantized V values are assumed to lie within the
 * f16 range (|v| <= 65504); the CUDA-core kernel has no such limit.
 */
int quant_sdpa_uses_tensor_cores(const ta_quant_params *p);

/*
 * Test hook, not for production use: quant_sdpa_fwd on the CUDA-core or the
 * warp-MMA kernel (p->kernel must resolve to one of them, else
 * TA_ERR_UNSUPPORTED) with the first K/V
 * copy wait of every CTA bounded by `first_wait_polls` polls instead of the
 * normal bound; 0 makes that wait give up at once.  It exercises the failure
 * path of the kernel's bounded waits without any fault: the CTA ORs 1 into the
 * status word (tmp's first 32-bit word), waits (with the normal bound) until
 * every copy it issued has landed, and returns.  The output is then not valid.
 * Same buffers and checks as quant_sdpa_fwd.
 */
ta_status ta_test_quant_sdpa_fwd_wait_limit(uint32_t first_wait_polls, const ta_quant_params *p,
                                            const ta_buf *queries, const ta_buf *k_packed,
                                            const ta_buf *k_scales, const ta_buf *k_biases,
                                            const ta_buf *v_packed, const ta_buf *v_scales,
                                            const ta_buf *v_biases, const ta_buf *sinks,
                                            const ta_buf *mask_bool, const ta_buf *mask_float,
                                            const ta_buf *tmp, const ta_buf *out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* TREE_ATTN_H_ */
