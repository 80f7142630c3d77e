"""Host-side checks of the C ABI: the library loads, exports every declared
symbol, sizes match the pages' numbers, and invalid calls fail before any
launch.  No call here reaches a kernel."""
import ctypes
import json
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tree_attn.h")


@pytest.fixture(scope="module")
def ta():
    from tree_masked_speculative_gb300 import build
    build.build()
    import tree_masked_speculative_gb300 as m
    return m


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\([^;{]*\)\s*;", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = _declared_functions()
    for n in ("tree_attn_fwd", "tree_attn_reduce", "quant_sdpa_fwd", "tree_attn_tmp_bytes",
              "ta_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(ta):
    for n in _declared_functions():
        assert hasattr(ta.lib, n), n
    # nothing but the ABI is exported from the .so (hidden visibility)
    out = os.popen("nm -D --defined-only %s" % ta.library_path()).read()
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert set(_declared_functions()) <= exported


def test_params_struct_is_36_bytes(ta):
    gold = json.load(open(os.path.join(ROOT, "tests", "golden", "tree_tmp_bytes.json")))
    assert ctypes.sizeof(ta.TreeParams) == gold["params_struct_bytes"]
    assert [f[0] for f in ta.TreeParams._fields_] == [
        "n_heads", "n_kv_heads", "head_dim", "kv_seq_len", "kv_capacity", "scale", "nwg", "q_l",
        "mask_stride"]


def test_tmp_bytes_matches_pages_example(ta):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "tree_tmp_bytes.json")))["tmp_bytes"]
    assert ta.tree_attn_tmp_bytes(g["n_heads"], g["head_dim"], g["q_l"], g["nwg"]) == g["bytes"]


def test_tmp_bytes_saturates(ta):
    big = 2 ** 32 - 1
    assert ta.tree_attn_tmp_bytes(big, big, big, big) == 2 ** 64 - 1
    assert ta.tree_attn_tmp_bytes(0, 256, 1, 32) == 0


def _p(ta, **kw):
    d = dict(n_heads=16, n_kv_heads=8, head_dim=256, kv_seq_len=100, kv_capacity=1024, scale=1.0,
             q_l=1, mask_stride=100, nwg=4)
    d.update(kw)
    return ta.tree_params(**d)


FAKE = 0x10000   # a 64 KiB-aligned address: validation never dereferences it


def _b(ta, nbytes, code, ptr=FAKE, reserved=0):
    return ta.Buf(ptr, nbytes, code, reserved)


def _tree_call(ta, p, q=None, k=None, v=None, mask=None, tmp=None, out=None):
    B = lambda n, c: _b(ta, n, c)
    H, L, D = p.n_heads, p.q_l, p.head_dim
    q = q or B(H * L * D * 4, ta.TA_F32)
    k = k or B(p.n_kv_heads * p.kv_capacity * D * 2, ta.TA_F16)
    v = v or B(p.n_kv_heads * p.kv_capacity * D * 2, ta.TA_F16)
    mask = mask or B(L * p.mask_stride * 4, ta.TA_F32)
    out = out or B(H * L * D * 4, ta.TA_F32)
    ws = ta.tree_attn_workspace_bytes(p)
    tmp = tmp or B(ws if ws < 2 ** 63 else 0, ta.TA_F32)
    before = ta.ta_launch_count()
    R = ctypes.byref
    st = ta.lib.tree_attn_fwd(ctypes.byref(p), R(q), R(k), R(v), R(mask), R(tmp), R(out), None)
    assert ta.ta_launch_count() == before, "a failing call must not launch"
    return st, ta.ta_last_error()


def test_validate_params_ok_cases(ta):
    # tree_attention.rs test_validate_params_ok and the head_dim 128 case
    assert ta.tree_attn_num_splits(_p(ta)) == 4
    assert ta.tree_attn_num_splits(_p(ta, n_heads=40, head_dim=128, kv_seq_len=64,
                                       kv_capacity=256, mask_stride=64)) == 4
    assert ta.tree_attn_workspace_bytes(_p(ta)) >= ta.tree_attn_tmp_bytes(16, 256, 1, 4)


def test_validate_mask_stride_too_small(ta):
    st, msg = _tree_call(ta, _p(ta, mask_stride=50))
    assert st == 1 and "mask_stride" in msg


def test_validate_bad_head_dim(ta):
    assert ta.tree_attn_num_splits(_p(ta, head_dim=64)) == 0
    st, msg = _tree_call(ta, _p(ta, head_dim=64))
    assert st == 1 and "head_dim" in msg


def test_validate_q_seq_len_zero(ta):
    st, msg = _tree_call(ta, _p(ta, q_l=0))
    assert st == 1 and "q_seq_len" in msg


@pytest.mark.parametrize("kw,frag", [
    (dict(n_heads=0), "num_heads"), (dict(n_kv_heads=0), "num_kv_heads"),
    (dict(n_heads=12, n_kv_heads=8), "divisible"), (dict(kv_seq_len=0), "kv_seq_len"),
    (dict(kv_capacity=99), "kv_capacity"), (dict(scale=float("nan")), "scale"),
])
def test_validate_params_rejections(ta, kw, frag):
    st, msg = _tree_call(ta, _p(ta, **kw))
    assert st == 1 and frag in msg


def test_validate_buffer_dtypes(ta):
    p = _p(ta)
    n = 1 << 30
    st, msg = _tree_call(ta, p, q=_b(ta, n, ta.TA_F16))
    assert st == 1 and "q dtype" in msg
    st, msg = _tree_call(ta, p, k=_b(ta, n, ta.TA_F16), v=_b(ta, n, ta.TA_BF16))
    assert st == 1 and "must match" in msg
    st, msg = _tree_call(ta, p, k=_b(ta, n, ta.TA_U32), v=_b(ta, n, ta.TA_U32))
    assert st == 1 and "F32, F16 or BF16" in msg
    st, msg = _tree_call(ta, p, mask=_b(ta, n, ta.TA_F16))
    assert st == 1 and "tree_mask dtype" in msg
    st, msg = _tree_call(ta, p, out=_b(ta, n, ta.TA_BF16))
    assert st == 1 and "output dtype" in msg
    st, msg = _tree_call(ta, p, tmp=_b(ta, n, ta.TA_F16))
    assert st == 1 and "tmp dtype" in msg


@pytest.mark.parametrize("which", ["q", "k", "v", "mask", "out", "tmp"])
def test_validate_undersized_buffers(ta, which):
    p = _p(ta)
    H, L, D = p.n_heads, p.q_l, p.head_dim
    need = {"q": (H * L * D * 4, ta.TA_F32), "k": (p.n_kv_heads * p.kv_capacity * D * 2, ta.TA_F16),
            "v": (p.n_kv_heads * p.kv_capacity * D * 2, ta.TA_F16),
            "mask": (L * p.mask_stride * 4, ta.TA_F32), "out": (H * L * D * 4, ta.TA_F32),
            "tmp": (ta.tree_attn_workspace_bytes(p), ta.TA_F32)}[which]
    st, msg = _tree_call(ta, p, **{which: _b(ta, need[0] - 1, need[1])})
    assert st == 2 and "too small" in msg


def test_validate_overflowing_sizes(ta):
    p = _p(ta, n_kv_heads=8, kv_capacity=2 ** 31 - 1, kv_seq_len=100, head_dim=512,
           n_heads=2 ** 16 * 8, q_l=2 ** 15 - 1)
    st, msg = _tree_call(ta, p, q=_b(ta, 2 ** 63, ta.TA_F32), out=_b(ta, 2 ** 63, ta.TA_F32))
    assert st in (2, 3, 4)


def test_validate_null_misaligned_and_reserved(ta):
    p = _p(ta)
    n = 1 << 30
    st, msg = _tree_call(ta, p, q=_b(ta, n, ta.TA_F32, ptr=0))
    # a NULL q with bytes > 0 is an error, not "absent"
    assert st == 1 and "NULL" in msg
    st, msg = _tree_call(ta, p, q=_b(ta, n, ta.TA_F32, ptr=FAKE + 4))
    assert st == 1 and "aligned" in msg
    st, msg = _tree_call(ta, p, q=_b(ta, n, ta.TA_F32, reserved=7))
    assert st == 1 and "reserved" in msg


def test_reduce_validates_before_launch(ta):
    p = _p(ta)
    before = ta.ta_launch_count()
    R = ctypes.byref
    st = ta.lib.tree_attn_reduce(ctypes.byref(p), R(_b(ta, 16, ta.TA_F32)), R(_b(ta, 1 << 30, ta.TA_F32)),
                                 None)
    assert st == 2 and ta.ta_launch_count() == before
    st = ta.lib.tree_attn_reduce(ctypes.byref(_p(ta, head_dim=96)), R(_b(ta, 1 << 30, ta.TA_F32)),
                                 R(_b(ta, 1 << 30, ta.TA_F32)), None)
    assert st == 1


@pytest.mark.parametrize("kw,pbytes,pdtype,st_want,frag", [
    (dict(q_l=10), 10 * 4, "U32", 1, "parents dtype"),
    (dict(q_l=10), None, None, 1, "parents is NULL"),                  # no parent array at all
    (dict(q_l=10), 9 * 4, "I32", 2, "parents"),
    (dict(q_l=120), 120 * 4, "I32", 1, "q_l"),                          # more nodes than keys
    (dict(q_l=257, kv_seq_len=1000, mask_stride=1000), 257 * 4, "I32", 4, "q_l <= 256"),
    (dict(q_l=10, head_dim=96), 10 * 4, "I32", 1, "head_dim"),
])
def test_tree_parents_rejections(ta, kw, pbytes, pdtype, st_want, frag):
    p = _p(ta, **kw)
    H, L, D = p.n_heads, p.q_l, p.head_dim
    B = lambda n, c: _b(ta, n, c)
    q, out = B(H * L * D * 4, ta.TA_F32), B(H * L * D * 4, ta.TA_F32)
    k = v = B(p.n_kv_heads * p.kv_capacity * D * 2, ta.TA_F16)
    ws = ta.tree_attn_workspace_bytes(p)
    tmp = B(ws if ws < 2 ** 63 else 0, ta.TA_F32)
    code = {"I32": ta.TA_I32, "U32": ta.TA_U32}
    R = ctypes.byref
    par = R(_b(ta, pbytes, code[pdtype])) if pbytes is not None else None
    before = ta.ta_launch_count()
    st = ta.lib.tree_attn_fwd_parents(R(p), par, R(q), R(k), R(v), R(tmp), R(out), None)
    assert ta.ta_launch_count() == before, "a failing call must not launch"
    assert st == st_want and frag in ta.ta_last_error()


def test_workspace_holds_ancestor_bitsets(ta):
    # a parent-array tree mask keeps q_l * ceil(q_l / 32) words of ancestor bits in tmp
    small = ta.tree_attn_workspace_bytes(_p(ta, q_l=32, kv_seq_len=1000, mask_stride=1000))
    large = ta.tree_attn_workspace_bytes(_p(ta, q_l=256, kv_seq_len=1000, mask_stride=1000))
    assert large - small >= 256 * 8 * 4 - 32 * 4


# ------------------------------------------------------------------- quant
def _qp(ta, **kw):
    d = dict(batch=2, n_q_heads=8, n_kv_heads=2, dim=128, tokens=100, bits=4, group_size=64,
             has_sinks=1, window_size=0, scale=0.1, nwg=3)
    d.update(kw)
    return ta.quant_params(**d)


def _quant_call(ta, p, T=None, **over):
    T = T if T is not None else ta.TA_F16
    rows, kvr = p.batch * p.n_q_heads, p.batch * p.n_kv_heads
    words = p.dim * p.bits // 32 if p.bits else 1
    groups = p.dim // p.group_size if p.group_size else 1
    bufs = dict(
        queries=_b(ta, rows * p.dim * 2, T),
        k_packed=_b(ta, kvr * p.tokens * words * 4, ta.TA_U32),
        k_scales=_b(ta, kvr * p.tokens * groups * 2, T), k_biases=_b(ta, kvr * p.tokens * groups * 2, T),
        v_packed=_b(ta, kvr * p.tokens * words * 4, ta.TA_U32),
        v_scales=_b(ta, kvr * p.tokens * groups * 2, T), v_biases=_b(ta, kvr * p.tokens * groups * 2, T),
        sinks=_b(ta, p.n_q_heads * 4, ta.TA_F32), mask_bool=ta.Buf(None, 0, ta.TA_U32, 0),
        mask_float=ta.Buf(None, 0, T, 0),
        tmp=_b(ta, max(0, ta.quant_sdpa_tmp_bytes(p)) if ta.quant_sdpa_tmp_bytes(p) < 2 ** 63 else 0,
               ta.TA_F32),
        out=_b(ta, rows * p.dim * 2, T))
    bufs.update(over)
    order = ["queries", "k_packed", "k_scales", "k_biases", "v_packed", "v_scales", "v_biases",
             "sinks", "mask_bool", "mask_float", "tmp", "out"]
    before = ta.ta_launch_count()
    st = ta.lib.quant_sdpa_fwd(ctypes.byref(p), *[ctypes.byref(bufs[k]) for k in order], None)
    assert ta.ta_launch_count() == before
    return st, ta.ta_last_error()


def test_quant_tmp_bytes(ta):
    p = _qp(ta)
    assert ta.quant_sdpa_num_splits(p) == 3
    assert ta.quant_sdpa_tmp_bytes(p) == 256 + 16 * 3 * (128 + 2) * 4
    assert ta.quant_sdpa_tmp_bytes(_qp(ta, nwg=1)) == 256


@pytest.mark.parametrize("kw,st_want,frag", [
    (dict(bits=3), 1, "bits"), (dict(dim=100), 1, "multiple of 32/bits"),
    (dict(group_size=48), 1, "group_size"), (dict(n_q_heads=6, n_kv_heads=4), 1, "divisible"),
    (dict(tokens=0), 1, "tokens"), (dict(has_sinks=2), 1, "has_sinks"),
    (dict(group_size=4), 4, "group_size"), (dict(dim=1024, group_size=64), 4, "dim"),
])
def test_quant_param_rejections(ta, kw, st_want, frag):
    st, msg = _quant_call(ta, _qp(ta, **kw))
    assert st == st_want and frag in msg


def test_quant_dtype_and_size_rejections(ta):
    p = _qp(ta)
    st, msg = _quant_call(ta, p, queries=_b(ta, 1 << 30, ta.TA_F32))
    assert st == 1 and "queries dtype" in msg
    st, msg = _quant_call(ta, p, k_scales=_b(ta, 1 << 30, ta.TA_BF16))
    assert st == 1 and "k_scales" in msg
    st, msg = _quant_call(ta, p, k_packed=_b(ta, 1 << 30, ta.TA_F32))
    assert st == 1 and "U32" in msg
    st, msg = _quant_call(ta, p, mask_float=_b(ta, 1 << 30, ta.TA_BF16))
    assert st == 1 and "mask_float" in msg
    st, msg = _quant_call(ta, p, out=_b(ta, 1 << 30, ta.TA_BF16))
    assert st == 1 and "out dtype" in msg
    st, msg = _quant_call(ta, p, v_packed=_b(ta, 16 * 100 * 4 - 4, ta.TA_U32))
    assert st == 2 and "v_packed" in msg
    st, msg = _quant_call(ta, p, mask_bool=_b(ta, 16 * 100 * 4 - 1, ta.TA_U32))
    assert st == 2 and "mask_bool" in msg
    st, msg = _quant_call(ta, p, tmp=_b(ta, 64, ta.TA_F32))
    assert st == 2 and "tmp" in msg


def test_kernel_choice_is_per_call(ta):
    """The kernel family travels with each call (no process-wide switch): an
    invalid choice is rejected before any launch, a valid one changes nothing
    for other calls."""
    d = dict(n_heads=4, n_kv_heads=2, head_dim=128, kv_seq_len=50, kv_capacity=64, scale=0.1, nwg=0, q_l=10,
             mask_stride=64)
    p = ta.TreeParams(**d)
    b = ctypes.byref(_b(ta, 1 << 30, ta.TA_F32))
    before = ta.ta_launch_count()
    for kernel, kind, frag in [(3, 0, "kernel"), (-1, 0, "kernel"), (0, 7, "mask_kind")]:
        o = ta.TreeOptions(kernel, kind, 0, 0)
        st = ta.lib.tree_attn_fwd_ex(ctypes.byref(p), ctypes.byref(o), b, b, b, b, b, b, None)
        assert st == 1 and frag in ta.ta_last_error()
    o = ta.TreeOptions(0, 0, 0, 5)
    assert ta.lib.tree_attn_fwd_ex(ctypes.byref(p), ctypes.byref(o), b, b, b, b, b, b, None) == 1
    assert "reserved" in ta.ta_last_error()
    assert ta.lib.tree_attn_fwd_ex(ctypes.byref(p), None, b, b, b, b, b, b, None) == 1
    o = ta.TreeOptions(0, ta.MASK_DENSE, 0, 0)
    assert ta.lib.tree_attn_fwd_ex(ctypes.byref(p), ctypes.byref(o), b, b, b, None, b, b, None) == 1
    assert "needs a mask" in ta.ta_last_error()
    q = ta.quant_params(1, 8, 2, 128, 100, 4, 64, 0, 0, 0.1, 0, 4)
    assert ta.quant_sdpa_uses_tensor_cores(q) == -1
    assert ta.quant_sdpa_tmp_bytes(q) == 2 ** 64 - 1
    assert ta.ta_launch_count() == before


def test_status_offset_is_the_workspace_header(ta):
    p = ta.tree_params(24, 4, 256, 4096, 8192, 1 / 16, 32, 4096, 5)
    ws = ta.tree_attn_workspace_bytes(p)
    off = ta.tree_attn_status_offset(p)
    assert off == ws - 256 and off % 256 == 0
    bad = ta.tree_params(24, 4, 100, 4096, 8192, 1 / 16, 32, 4096, 5)
    assert ta.tree_attn_status_offset(bad) == 2 ** 64 - 1


# ------------------------------------------------------------ tree mask builder
@pytest.mark.parametrize("kw,pbytes,pdtype,mbytes,mdtype,st_want,frag", [
    (dict(), 10 * 4, "I32", 10 * 64 * 4, "F32", None, None),                 # valid shape; see below
    (dict(), 10 * 4, "U32", 10 * 64 * 4, "F32", 1, "parents dtype"),
    (dict(), 10 * 4, "I32", 10 * 64 * 4, "F16", 1, "mask dtype"),
    (dict(), 9 * 4, "I32", 10 * 64 * 4, "F32", 2, "parents"),
    (dict(), 10 * 4, "I32", 10 * 64 * 4 - 4, "F32", 2, "mask"),
    (dict(mask_stride=40), 10 * 4, "I32", 10 * 64 * 4, "F32", 1, "mask_stride"),
    (dict(q_l=60, kv_seq_len=50, mask_stride=64), 60 * 4, "I32", 60 * 64 * 4, "F32", 1, "q_l"),
    (dict(q_l=16385, kv_seq_len=20000, mask_stride=20000), 16385 * 4, "I32", 16385 * 20000 * 4, "F32", 4, "q_l"),
])
def test_tree_mask_build_rejections(ta, kw, pbytes, pdtype, mbytes, mdtype, st_want, frag):
    if st_want is None:
        return                                               # launching needs a GPU (tests/test_gpu_tree.py)
    d = dict(n_heads=4, n_kv_heads=2, head_dim=128, kv_seq_len=50, kv_capacity=64, scale=0.1, nwg=0, q_l=10,
             mask_stride=64)
    d.update(kw)
    d["kv_capacity"] = max(d["kv_capacity"], d["kv_seq_len"])
    p = ta.TreeParams(**d)
    code = {"I32": ta.TA_I32, "U32": ta.TA_U32, "F32": ta.TA_F32, "F16": ta.TA_F16}
    before = ta.ta_launch_count()
    st = ta.lib.tree_mask_build(ctypes.byref(p), ctypes.byref(_b(ta, pbytes, code[pdtype])),
                                ctypes.byref(_b(ta, mbytes, code[mdtype])), None)
    assert ta.ta_launch_count() == before
    assert st == st_want and frag in ta.ta_last_error()


def test_quant_kernel_family_choice(ta):
    """Which quantized kernel a shape takes (no device work)."""
    def p(dim, G=64, nQ=32, nKV=8, bits=4, kernel=0):
        return ta.quant_params(1, nQ, nKV, dim, 1000, bits, G, 0, 0, 0.1, 0, kernel)
    fam = ta.quant_sdpa_kernel_family
    TC, MMA, CC = ta.KERNEL_TENSOR_CORES, ta.KERNEL_WARP_MMA, ta.KERNEL_CUDA_CORES
    assert fam(p(128)) == MMA                 # 4 rows per KV row: warp MMA
    assert fam(p(128, nQ=128)) == MMA         # 16 rows per KV row, dim 128: the warp-MMA wide form
    assert fam(p(64, G=32, nQ=256)) == MMA    # 32 rows per KV row, dim 64
    assert fam(p(256, nQ=128)) == TC          # 16 rows per KV row, dim 256: tcgen05
    assert fam(p(128, G=128, nQ=128)) == TC   # group size 128: tcgen05
    assert fam(p(512, nQ=256)) == CC          # neither tensor-core kernel takes dim 512
    assert fam(p(96, G=32)) == CC             # warp MMA: dims 64, 128, 256 only
    assert fam(p(128, G=128)) == CC           # warp MMA: group size 32 or 64 only
    assert fam(p(256, bits=8)) == MMA
    assert fam(p(256, bits=8, nQ=256)) == MMA  # tcgen05 rings exceed shared memory: warp MMA
    assert fam(p(64, G=32, bits=8)) == MMA
    assert fam(p(128, kernel=1)) == CC
    assert fam(p(128, kernel=3)) == MMA
    assert fam(p(128, nQ=128, kernel=3)) == MMA
    assert fam(p(512, kernel=3)) == CC
    assert fam(p(128, kernel=2)) == TC
    assert fam(p(256, bits=4, kernel=2)) == TC
    assert fam(p(256, bits=8, kernel=2)) == CC        # rings exceed shared memory
    assert fam(p(64, G=32, kernel=2)) == TC
    assert fam(p(512, kernel=2)) == CC                # O alone fills TMEM
    assert fam(p(96, G=32, kernel=2)) == CC           # not a multiple of 64
    assert fam(p(256, G=16, nQ=256, bits=8, kernel=2)) == CC   # 16 groups x 32 rows
    assert fam(p(100)) == -1                  # invalid params
    assert fam(p(128, kernel=4)) == -1        # no such family
    assert ta.quant_sdpa_uses_tensor_cores(p(128)) == 1
    assert ta.quant_sdpa_uses_tensor_cores(p(128, kernel=1)) == 0
    assert ta.quant_sdpa_uses_tensor_cores(p(512, nQ=256)) == 0
    assert ta.quant_sdpa_uses_tensor_cores(p(100)) == -1


@pytest.mark.parametrize("q_l,nQ,tokens,pbytes,pdtype,st_want,frag", [
    (0, 8, 100, 64, "I32", 1, "q_l must be > 0"),
    (33, 66, 100, 33 * 4, "I32", 4, "<= 32"),
    (8, 12, 100, 32, "I32", 1, "multiple of q_l"),
    (8, 16, 5, 32, "I32", 1, "<= tokens"),
    (8, 16, 100, 32, "U32", 1, "parents dtype"),
    (8, 16, 100, 28, "I32", 2, "parents"),
    (8, 16, 100, None, None, 1, "parents is NULL"),
])
def test_quant_tree_rejections(ta, q_l, nQ, tokens, pbytes, pdtype, st_want, frag):
    """quant_sdpa_fwd_tree's own checks, before any launch."""
    p = ta.quant_params(1, nQ, 2, 128, tokens, 4, 64, 0, 0, 0.1, 1, 1)
    B = lambda n, c: ctypes.byref(_b(ta, n, c))
    big = 1 << 30
    code = {"I32": ta.TA_I32, "U32": ta.TA_U32}
    par = B(pbytes, code[pdtype]) if pbytes is not None else None
    before = ta.ta_launch_count()
    st = ta.lib.quant_sdpa_fwd_tree(ctypes.byref(p), q_l, par, B(big, ta.TA_F16), B(big, ta.TA_U32),
                                    B(big, ta.TA_F16), B(big, ta.TA_F16), B(big, ta.TA_U32), B(big, ta.TA_F16),
                                    B(big, ta.TA_F16), None, None, B(big, ta.TA_F32), B(big, ta.TA_F16), None)
    assert ta.ta_launch_count() == before
    assert st == st_want and frag in ta.ta_last_error(), ta.ta_last_error()
