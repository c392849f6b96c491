"""Host-side validation through pa_varlen_check (no GPU, no CUDA call).

The cases come from the candle error-explanation pages (tests/golden/validation_cases.json,
each with its citation); the descriptors point at fake, 16-byte aligned addresses because
the check never dereferences them."""
import json
import os

import pytest

from paged_kv_varlen_flashattention_gb300 import binding

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "validation_cases.json")
CASES = json.load(open(GOLDEN))["cases"]
CODES = {v: k for k, v in binding.STATUS.items()}


def contiguous(shape):
    st, acc = [], 1
    for s in reversed(shape):
        st.append(acc)
        acc *= s
    return list(reversed(st))


def desc(shape, dtype, stride=None, addr=0x100000):
    d = binding.PaTensor()
    d.data = addr
    d.dtype = dtype
    d.ndim = len(shape)
    for i, s in enumerate(shape):
        d.shape[i] = s
    for i, s in enumerate(stride or contiguous(shape)):
        d.stride[i] = s
    return d


def build(case):
    q = case.get("q", [8, 4, 64])
    k = case.get("k", [6, 32, 2, 64])
    v = case.get("v", [6, 32, 2, 64])
    out = case.get("out", q if len(q) == 3 else [8, 4, 64])
    bt = case.get("block_table", [2, 3])
    H = q[-2] if len(q) >= 2 else 4
    D = case.get("head_dim", q[-1])
    Hkv = k[-2]
    P = case.get("page_block_size", 32)
    ds = [
        desc(q, binding.PA_BF16, case.get("q_stride")),
        desc(k, binding.PA_BF16, case.get("k_stride")),
        desc(v, binding.PA_BF16, case.get("v_stride")),
        desc([3], binding.PA_I32, case.get("cu_q_stride")),
        desc([3], binding.PA_I32, case.get("cu_k_stride")),
        None if bt is None else desc(bt, binding.PA_I32, case.get("bt_stride")),
        desc(out, binding.PA_BF16),
        desc([4, 8], binding.PA_F32),
    ]
    return ds, H, Hkv, D, (P if bt is not None else 0)


def run_check(ds, H, Hkv, D, P, max_sq=5, max_sk=64, wl=-1, wr=0, scale=0.125):
    lib = binding.load()
    r = lambda d: None if d is None else binding.ctypes.byref(d)  # noqa: E731
    rc = lib.pa_varlen_check(r(ds[0]), r(ds[1]), r(ds[2]), r(ds[3]), r(ds[4]), r(ds[5]), max_sq, max_sk, H, Hkv,
                             D, P, scale, wl, wr, r(ds[6]), r(ds[7]))
    return rc, lib.pa_last_error().decode()


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_page_case(case):
    ds, H, Hkv, D, P = build(case)
    rc, msg = run_check(ds, H, Hkv, D, P)
    assert binding.STATUS[rc] == case["expect"], (msg, case["citation"])
    if "message" in case:
        assert case["message"] in msg, msg
    if rc == 0:
        assert msg == ""


def _base():
    return build({})


def test_scalar_disagreement_is_an_argument_error():
    ds, H, Hkv, D, P = _base()
    assert run_check(ds, H + 1, Hkv, D, P)[0] == CODES["PA_ERR_ARG"]
    assert run_check(ds, H, Hkv, D + 8, P)[0] == CODES["PA_ERR_ARG"]
    assert run_check(ds, H, Hkv + 1, D, P)[0] == CODES["PA_ERR_ARG"]


def test_gqa_divisibility():
    ds, _, _, D, P = build({"q": [8, 3, 64], "out": [8, 3, 64]})
    ds[7] = desc([3, 8], binding.PA_F32)
    rc, msg = run_check(ds, 3, 2, D, P)
    assert rc == CODES["PA_ERR_ARG"] and "multiple of num_heads_k" in msg


def test_dtype_rules():
    ds, H, Hkv, D, P = _base()
    ds[1] = desc([6, 32, 2, 64], binding.PA_F16)
    assert run_check(ds, H, Hkv, D, P)[0] == CODES["PA_ERR_ARG"]
    ds, H, Hkv, D, P = _base()
    ds[7] = desc([4, 8], binding.PA_BF16)
    assert run_check(ds, H, Hkv, D, P)[0] == CODES["PA_ERR_ARG"]
    ds, H, Hkv, D, P = _base()
    ds[3] = desc([3], binding.PA_F32)
    assert run_check(ds, H, Hkv, D, P)[0] == CODES["PA_ERR_ARG"]
    ds, H, Hkv, D, P = _base()
    for i in (0, 1, 2, 6):
        ds[i].dtype = binding.PA_F32
    assert run_check(ds, H, Hkv, D, P)[0] == CODES["PA_ERR_UNSUPPORTED"]


def test_out_and_lse_shapes():
    ds, H, Hkv, D, P = _base()
    ds[6] = desc([8, 4, 32], binding.PA_BF16)
    assert run_check(ds, H, Hkv, D, P)[0] == CODES["PA_ERR_ARG"]
    ds, H, Hkv, D, P = _base()
    ds[7] = desc([8, 4], binding.PA_F32)
    assert run_check(ds, H, Hkv, D, P)[0] == CODES["PA_ERR_ARG"]


def test_block_table_rows_and_width():
    ds, H, Hkv, D, P = _base()
    ds[5] = desc([3, 3], binding.PA_I32)
    assert run_check(ds, H, Hkv, D, P)[0] == CODES["PA_ERR_ARG"]
    ds, H, Hkv, D, P = _base()
    rc, msg = run_check(ds, H, Hkv, D, P, max_sk=97)  # 3 pages of 32 hold 96 keys
    assert rc == CODES["PA_ERR_ARG"] and "too few for max_seqlen_k" in msg
    assert run_check(ds, H, Hkv, D, P, max_sk=96)[0] == 0


def test_implementation_limits():
    ds, H, Hkv, D, P = build({"q": [8, 4, 60], "k": [6, 32, 2, 60], "v": [6, 32, 2, 60], "out": [8, 4, 60]})
    rc, msg = run_check(ds, H, Hkv, 60, P)
    assert rc == CODES["PA_ERR_UNSUPPORTED"] and "multiple of 8" in msg
    ds, H, Hkv, D, P = _base()
    ds[0].data = 0x100008  # not 16-byte aligned
    assert run_check(ds, H, Hkv, D, P)[0] == CODES["PA_ERR_UNSUPPORTED"]
    ds, H, Hkv, D, P = _base()
    ds[0].stride[0] = 260  # not a multiple of 8 elements
    assert run_check(ds, H, Hkv, D, P)[0] == CODES["PA_ERR_UNSUPPORTED"]


def test_grid_limit_of_long_rows():
    """Long query rows the tensor-core prefill kernel does not take (head_dim 512 here) are
    split-KV row tiles of 32 rows: num_heads_k x tiles must fit the 65,535 CTAs of grid.y."""
    shp = {"q": [8, 4, 512], "k": [6, 32, 2, 512], "v": [6, 32, 2, 512], "out": [8, 4, 512]}
    ds, H, Hkv, D, P = build(shp)
    rc, msg = run_check(ds, H, Hkv, D, P, max_sq=300000)  # 600,000 rows -> 18,750 tiles x 2 kv heads
    assert rc == 0, msg
    rc, msg = run_check(ds, H, Hkv, D, P, max_sq=600000)  # 37,500 tiles x 2 kv heads > 65,535
    assert rc == CODES["PA_ERR_UNSUPPORTED"] and "65535" in msg, msg
    ds, H, Hkv, D, P = _base()  # head_dim 64, G = 2: the tensor-core prefill takes the long rows
    assert run_check(ds, H, Hkv, D, P, max_sq=600000)[0] == 0


def test_non_finite_scale():
    ds, H, Hkv, D, P = _base()
    assert run_check(ds, H, Hkv, D, P, scale=float("nan"))[0] == CODES["PA_ERR_ARG"]


def test_check_order_follows_the_pages():
    """Several faults at once: the rank fault is reported before contiguity, contiguity
    before shapes, shapes before the page size, the page size before the head size."""
    ds, H, Hkv, D, P = build({"k": [192, 2, 64], "v": [192, 2, 64], "q_stride": [512, 128, 2]})
    assert run_check(ds, H, Hkv, D, P)[0] == CODES["PA_ERR_RANK_PAGED"]
    ds, H, Hkv, D, P = build({"q_stride": [512, 128, 2], "v": [6, 32, 1, 64]})
    assert run_check(ds, H, Hkv, D, P)[0] == CODES["PA_ERR_NONCONTIG"]
    ds, H, Hkv, D, P = build({"v": [6, 32, 1, 64], "page_block_size": 0})
    assert run_check(ds, H, Hkv, D, P)[0] == CODES["PA_ERR_SHAPE"]
    ds, H, Hkv, D, P = build({"q": [8, 4, 576], "k": [6, 16, 2, 576], "v": [6, 16, 2, 576], "out": [8, 4, 576],
                              "head_dim": 576, "page_block_size": 16})
    assert run_check(ds, H, Hkv, D, P)[0] == CODES["PA_ERR_PAGE_MULT32"]


def run_check_alibi(ds, alibi, H, Hkv, D, P, max_sq=5, max_sk=64, wl=-1, wr=0, scale=0.125):
    lib = binding.load()
    r = lambda d: None if d is None else binding.ctypes.byref(d)  # noqa: E731
    rc = lib.pa_varlen_check_alibi(r(ds[0]), r(ds[1]), r(ds[2]), r(ds[3]), r(ds[4]), r(ds[5]), max_sq, max_sk, H,
                                   Hkv, D, P, scale, wl, wr, r(alibi), r(ds[6]), r(ds[7]))
    return rc, lib.pa_last_error().decode()


def test_alibi_slopes_checks():
    """alibi_slopes: one f32 slope per query head.  The shape condition carries the text of
    the "shape mismatch alibi_slopes {:?}, expected {:?}" related error of "paged flash-attn
    requires page_block_size to be a multiple of 32"; NULL behaves as pa_varlen_check."""
    ds, H, Hkv, D, P = _base()
    assert run_check_alibi(ds, None, H, Hkv, D, P) == run_check(ds, H, Hkv, D, P)
    assert run_check_alibi(ds, desc([H], binding.PA_F32), H, Hkv, D, P)[0] == 0
    for bad in ([H + 1], [H - 1], [1, H], [H, 1]):
        rc, msg = run_check_alibi(ds, desc(bad, binding.PA_F32), H, Hkv, D, P)
        assert rc == CODES["PA_ERR_SHAPE"] and "shape mismatch alibi_slopes" in msg and f"expected [{H}]" in msg
    rc, msg = run_check_alibi(ds, desc([H], binding.PA_F32, [2]), H, Hkv, D, P)
    assert rc == CODES["PA_ERR_NONCONTIG"] and "alibi_slopes" in msg
    rc, msg = run_check_alibi(ds, desc([H], binding.PA_BF16), H, Hkv, D, P)
    assert rc == CODES["PA_ERR_ARG"] and "alibi_slopes must be f32" in msg
    # the q/k/v conditions of the pages come first: a rank error wins over a bad alibi shape
    bad_q = list(ds)
    bad_q[0] = desc([8, 4, 64, 1], binding.PA_BF16)
    assert run_check_alibi(bad_q, desc([H + 1], binding.PA_F32), H, Hkv, D, P)[0] == CODES["PA_ERR_RANK"]


def _append_descs(**over):
    """Descriptors of a valid pa_kv_append call: 10 new tokens, 2 sequences, a (6, 32, 2, 64)
    pool, bf16."""
    shapes = {"k_new": [10, 2, 64], "v_new": [10, 2, 64], "cu_new": [3], "cu_k": [3], "bt": [2, 3],
              "k": [6, 32, 2, 64], "v": [6, 32, 2, 64]}
    dtypes = {"k_new": binding.PA_BF16, "v_new": binding.PA_BF16, "cu_new": binding.PA_I32,
              "cu_k": binding.PA_I32, "bt": binding.PA_I32, "k": binding.PA_BF16, "v": binding.PA_BF16}
    strides = {}
    for key, val in over.items():
        name, what = key.rsplit("_", 1) if key.endswith(("_shape", "_dtype", "_stride")) else (key, None)
        {"shape": shapes, "dtype": dtypes, "stride": strides}[what][name] = val
    order = ["k_new", "v_new", "cu_new", "cu_k", "bt", "k", "v"]
    return [desc(shapes[n], dtypes[n], strides.get(n)) for n in order]


def append_check(P=32, **over):
    rc = binding.kv_append_check(_append_descs(**over), P)
    return binding.STATUS[rc], binding.load().pa_last_error().decode()


def test_kv_append_checks():
    """pa_kv_append's host checks reuse the pages' conditions for the paged caches (rank 4,
    last-dim contiguity, k/v shapes, page size, head size), in the pages' order."""
    assert append_check() == ("PA_OK", "")
    st, msg = append_check(k_new_shape=[10, 2, 64, 1])
    assert st == "PA_ERR_RANK" and "rank 3" in msg
    st, msg = append_check(k_shape=[6 * 32, 2, 64], v_shape=[6 * 32, 2, 64])
    assert st == "PA_ERR_RANK_PAGED" and "paged expects k/v tensors of rank 4" in msg
    st, msg = append_check(k_stride=[32 * 2 * 64, 2 * 64, 64, 2])
    assert st == "PA_ERR_NONCONTIG" and "contiguous" in msg
    st, msg = append_check(v_shape=[6, 32, 2, 72])
    assert st == "PA_ERR_SHAPE" and "shape mismatch k" in msg
    st, msg = append_check(k_new_shape=[10, 1, 64], v_new_shape=[10, 1, 64])
    assert st == "PA_ERR_SHAPE" and "k_new" in msg
    assert append_check(P=0)[0] == "PA_ERR_PAGE_UNSET"
    st, msg = append_check(P=64)
    assert st == "PA_ERR_PAGE_MISMATCH" and "does not match k shape" in msg
    assert append_check(P=48, k_shape=[6, 48, 2, 64], v_shape=[6, 48, 2, 64])[0] == "PA_ERR_PAGE_MULT32"
    big = [6, 32, 2, 520]
    assert append_check(k_shape=big, v_shape=big, k_new_shape=[10, 2, 520], v_new_shape=[10, 2, 520])[0] \
        == "PA_ERR_HEADDIM"
    assert append_check(cu_k_shape=[4])[0] == "PA_ERR_ARG"
    assert append_check(bt_shape=[3, 3])[0] == "PA_ERR_ARG"
    assert append_check(bt_stride=[1, 2])[0] == "PA_ERR_NONCONTIG"
    assert append_check(v_new_dtype=binding.PA_F16)[0] == "PA_ERR_ARG"
    assert append_check(cu_new_dtype=binding.PA_F32)[0] == "PA_ERR_ARG"
    assert append_check(k_new_stride=[2 * 64 + 4, 64, 1])[0] == "PA_ERR_UNSUPPORTED"
    # a strided view of new tokens (e.g. K rows of a fused projection output) is fine
    assert append_check(k_new_stride=[3 * 2 * 64, 64, 1])[0] == "PA_OK"



def _padded(q=(2, 7, 4, 64), k=(2, 9, 2, 64), v=None, out=None, lse=None, alibi=None, q_stride=None,
            dtype=binding.PA_BF16):
    v = v or k
    out = out or q
    lse = lse or (q[0], q[2], q[1])
    return [desc(list(q), dtype, q_stride), desc(list(k), dtype), desc(list(v), dtype),
            None if alibi is None else desc(list(alibi), binding.PA_F32), desc(list(out), dtype),
            desc(list(lse), binding.PA_F32)]


def padded_status(ds, H=4, Hkv=2, D=64):
    rc = binding.check_padded(ds, H, Hkv, D)
    return binding.STATUS[rc], binding.load().pa_last_error().decode()


def test_padded_checks():
    """pa_check_padded: rank 4 inputs ("use FlashAttention (non-varlen) for padded batch
    attention", the Solutions of "flash-attn-varlen expects input tensors of rank 3"), then
    the varlen call's checks on the packed view."""
    assert padded_status(_padded()) == ("PA_OK", "")
    assert padded_status(_padded(alibi=(4,)))[0] == "PA_OK"
    st, msg = padded_status(_padded(q=(14, 4, 64), out=(14, 4, 64), lse=(2, 4, 7)))
    assert st == "PA_ERR_RANK" and "rank 4" in msg
    st, msg = padded_status(_padded(v=(2, 9, 2, 72)))
    assert st == "PA_ERR_SHAPE" and "shape mismatch k" in msg
    st, msg = padded_status(_padded(k=(3, 9, 2, 64)))
    assert st == "PA_ERR_SHAPE" and "shape mismatch q" in msg
    assert padded_status(_padded(alibi=(5,)))[0] == "PA_ERR_SHAPE"
    assert padded_status(_padded(lse=(2, 7, 4)))[0] == "PA_ERR_ARG"
    assert padded_status(_padded(q_stride=[7 * 4 * 64 + 8, 4 * 64, 64, 1]))[0] == "PA_ERR_UNSUPPORTED"
    assert padded_status(_padded(), H=5)[0] == "PA_ERR_ARG"
    assert padded_status(_padded(q_stride=[7 * 4 * 64, 4 * 64, 64, 2]))[0] == "PA_ERR_NONCONTIG"
