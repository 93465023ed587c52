"""Host-side tests of the C ABI that need no GPU: the library loads, exports
every entry point its header declares, and rejects bad arguments before any
launch (so no device memory is touched; the pointers below are never
dereferenced)."""
import ctypes
import os
import re

import pytest

import shared_kv_cache_gb300 as gqa
from shared_kv_cache_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gqa.load_library()


def header_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(gqa_[a-z_0-9]+)\s*\(", text))
    return names


def test_exports_every_declared_symbol(lib):
    declared = header_functions()
    assert {"gqa_forward", "gqa_workspace_size", "gqa_check_device_status", "gqa_status_string"} <= declared
    for name in declared:
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for code, name in [(0, "GQA_OK"), (1, "GQA_ERR_INVALID_ARGUMENT"), (2, "GQA_ERR_KV_OVERFLOW"),
                       (3, "GQA_ERR_UNSUPPORTED"), (4, "GQA_ERR_CUDA"), (5, "GQA_ERR_TIMEOUT")]:
        assert gqa.gqa_status_string(code) == name


# fake, 16-byte aligned device addresses: every call below fails validation first
P = {n: 0x10000 * (i + 1) for i, n in enumerate(
    ["q", "k", "v", "kb", "vb", "seq", "cos", "sin", "bias", "out", "ws"])}


def call(dims, total=64, **over):
    a = dict(query=P["q"], key=P["k"], value=P["v"], past_key=P["kb"], past_value=P["vb"],
             present_key=P["kb"], present_value=P["vb"], seqlens_k=P["seq"], total_sequence_length=total,
             cos_cache=P["cos"], sin_cache=P["sin"], scale=0.0, local_window_size=0, attention_bias=None,
             output=P["out"], workspace=P["ws"], workspace_bytes=1 << 30)
    a.update(over)
    return gqa.gqa_forward(dims, **a)


def dims(**over):
    d = dict(batch=2, seq_len=4, num_heads=8, kv_num_heads=2, head_size=64, max_seq_len=128, dtype="fp16",
             rotary_interleaved=0, cos_cache_rows=128, bias_batch=1, bias_heads=1)
    d.update(over)
    return gqa.make_dims(**d)


@pytest.mark.parametrize("bad", [
    dict(batch=0), dict(seq_len=0), dict(num_heads=6, kv_num_heads=4), dict(head_size=12),
    dict(head_size=264), dict(head_size=0), dict(max_seq_len=0), dict(dtype=7), dict(rotary_interleaved=2),
    dict(kv_num_heads=0), dict(kv_eviction=2),
])
def test_bad_dims_rejected(lib, bad):
    assert call(dims(**bad)) == gqa.GQA_ERR_INVALID_ARGUMENT


def test_overflow_rejected_before_launch(lib):
    # total_sequence_length beyond the buffer: the operator fails
    assert call(dims(max_seq_len=128), total=129) == gqa.GQA_ERR_KV_OVERFLOW
    assert call(dims(max_seq_len=4096, seq_len=128), total=4128) == gqa.GQA_ERR_KV_OVERFLOW


def test_binding_checks(lib):
    """Shared binding (both pairs equal) or non-shared (four distinct
    buffers); every call below breaks a rule and is rejected before any
    launch."""
    PK, PV = 0x200000, 0x300000   # separate present buffers (fake addresses)
    # one pair shared and the other not
    assert call(dims(), present_key=P["kb"] + 4096) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert call(dims(), present_value=P["vb"] + 4096) == gqa.GQA_ERR_INVALID_ARGUMENT
    ns = dict(present_key=PK, present_value=PV)
    # a past buffer that is another buffer of the call
    assert call(dims(past_seq_len=64), past_key=PV, **ns) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert call(dims(past_seq_len=64), past_value=PK, **ns) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert call(dims(past_seq_len=64), past_value=P["kb"], **ns) == gqa.GQA_ERR_INVALID_ARGUMENT
    # the past's slot count outside [0, M]
    assert call(dims(past_seq_len=129, max_seq_len=128), **ns) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert call(dims(past_seq_len=-1), **ns) == gqa.GQA_ERR_INVALID_ARGUMENT
    # a misaligned past buffer
    assert call(dims(past_seq_len=64), past_key=P["kb"] + 8, **ns) == gqa.GQA_ERR_INVALID_ARGUMENT


def test_pointer_checks(lib):
    # packed QKV (key and value both NULL) passes the pointer checks: the
    # call fails only at the later scale check
    assert call(dims(), key=None, value=None, scale=float("nan")) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert call(dims(), key=None, value=None, query=P["q"] + 2) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert call(dims(), key=None) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert call(dims(), value=None) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert call(dims(), query=None) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert call(dims(), output=None) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert call(dims(), seqlens_k=None) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert call(dims(), query=P["q"] + 2) == gqa.GQA_ERR_INVALID_ARGUMENT          # misaligned
    assert call(dims(), sin_cache=None) == gqa.GQA_ERR_INVALID_ARGUMENT            # half a rotary pair
    assert call(dims(), present_value=P["kb"], past_value=P["kb"]) == gqa.GQA_ERR_INVALID_ARGUMENT


def test_length_and_cache_checks(lib):
    assert call(dims(seq_len=8), total=7) == gqa.GQA_ERR_INVALID_ARGUMENT         # total < S
    assert call(dims(cos_cache_rows=32), total=64) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert call(dims(bias_batch=3), attention_bias=P["bias"]) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert call(dims(bias_heads=2), attention_bias=P["bias"]) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert call(dims(), scale=float("nan")) == gqa.GQA_ERR_INVALID_ARGUMENT


def test_workspace_checks(lib):
    d = dims()
    need = gqa.gqa_workspace_size(d, 64, 0)
    assert need > 0
    assert call(d, workspace_bytes=need - 1) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert call(d, workspace=None) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert gqa.gqa_workspace_size(dims(batch=0), 64, 0) == 0


def test_workspace_plan_decode(lib):
    # decode at D = 128: 2 * 2 partial slots per persistent CTA (one or two
    # CTAs per SM on 152 SMs), each G x (D + 2) fp32 values plus an 8-byte
    # arrival counter, and the 8-byte chunk ticket -- whatever the lengths
    d = dims(seq_len=1, head_size=128, num_heads=32, kv_num_heads=8, batch=16, max_seq_len=4096)
    big = gqa.gqa_workspace_size(d, 4096, 0)
    assert big > 0 and big % 256 == 0
    assert gqa.gqa_workspace_size(d, 17, 0) == big == gqa.gqa_workspace_size(d, 4096, 100)
    per_slot = 4 * 130 * 4 + 8
    assert big >= 4 * 152 * per_slot and big <= 4 * 2 * 152 * per_slot + 8 + 3 * 256


def call_host(dims, total=64, **over):
    a = dict(query=P["q"], key=P["k"], value=P["v"], past_key=P["kb"], past_value=P["vb"],
             present_key=P["kb"], present_value=P["vb"], seqlens_k=P["seq"], total_sequence_length=total,
             cos_cache=P["cos"], sin_cache=P["sin"], scale=0.0, local_window_size=0, attention_bias=None,
             output=P["out"], workspace=P["ws"], workspace_bytes=1 << 30)
    a.update(over)
    return gqa.gqa_forward_host(dims, **a)


def test_host_entry_workspace_and_checks(lib):
    # gqa_forward's scratch rounded to 256, then query, key, value, seqlens_k
    # and output copies, each rounded to 256 bytes
    d = dims()  # B 2, S 4, H 8, Hkv 2, D 64, fp16
    base = gqa.gqa_workspace_size(d, 64, 0)
    qb, kb, sb = 2 * 4 * 8 * 64 * 2, 2 * 4 * 2 * 64 * 2, 2 * 4
    r = lambda x: (x + 255) // 256 * 256  # noqa: E731
    need = gqa.gqa_workspace_size_host(d, 64, 0)
    assert need == r(base) + 2 * r(qb) + 2 * r(kb) + r(sb)
    assert gqa.gqa_workspace_size_host(dims(batch=0), 64, 0) == 0
    assert gqa.gqa_workspace_size_host(dims(seq_len=8), 7, 0) == 0
    # checks the host can make come first, in gqa_forward's order
    assert call_host(dims(batch=0)) == gqa.GQA_ERR_INVALID_ARGUMENT
    # packed QKV is a valid form here too: these fake addresses fail only as
    # memory that is not page-locked (before any launch)
    assert call_host(d, key=None, value=None, workspace_bytes=need) == gqa.GQA_ERR_INVALID_ARGUMENT
    for bad in (dict(query=None), dict(output=None), dict(seqlens_k=None), dict(key=None), dict(value=None),
                dict(query=P["q"] + 8), dict(seqlens_k=P["seq"] + 2), dict(workspace=None),
                dict(workspace_bytes=need - 1), dict(workspace=P["ws"] + 8)):
        assert call_host(d, **{"workspace_bytes": need, **bad}) == gqa.GQA_ERR_INVALID_ARGUMENT, bad
    # the fake addresses are not page-locked host memory: rejected before any launch
    assert call_host(d, workspace_bytes=need) == gqa.GQA_ERR_INVALID_ARGUMENT


def _r256(x):
    return (x + 255) // 256 * 256


def test_workspace_plan_generic_path():
    # head size other than 128: the append kernel writes the rotated queries
    # to the workspace, T [B, S, H, D]
    d = dims(batch=3, seq_len=5, num_heads=8, kv_num_heads=2, head_size=64, max_seq_len=256)
    assert gqa.gqa_workspace_size(d, 205, 0) == _r256(3 * 5 * 8 * 64 * 2)


def test_workspace_plan_prefill_splits():
    # tensor-core prefill, one query head per CTA and two CTAs per SM: a grid
    # of at least two CTAs per CTA slot (B * H * query tiles >= 2 * 2 * 152)
    # needs no scratch
    big = dims(batch=4, seq_len=2048, num_heads=32, kv_num_heads=8, head_size=128, max_seq_len=4096)
    assert gqa.gqa_workspace_size(big, 2048, 0) == 0
    # a smaller grid cuts each item's key range into at most
    # max(2, min(ceil(3 * 304 / items), 64-key tiles + 1)) pieces and keeps
    # fp32 partials (rows = items x pieces x 128 rows; D floats plus a
    # 16-byte (m, l) record each), after the work list: a 16-byte header, one
    # 16-byte entry per CTA of the grid (min(items x pieces, 2 x 304 +
    # items)) and two ints per item (its piece count and arrival count)
    small = dims(batch=8, seq_len=128, num_heads=32, kv_num_heads=8, head_size=128, max_seq_len=4096)
    items = 8 * 32 * 1
    pieces = min(-(-3 * 304 // items), 4096 // 64 + 1)
    assert pieces == 4
    rows = items * pieces * 128
    sched = _r256(16 + min(items * pieces, 304 * 2 + items) * 16 + items * 8)
    assert gqa.gqa_workspace_size(small, 4096, 0) == _r256(sched + _r256(rows * 128 * 4) + rows * 4 * 4)
    # few key tiles bound the pieces
    short = dims(batch=1, seq_len=128, num_heads=8, kv_num_heads=8, head_size=128, max_seq_len=4096)
    items = 1 * 8 * 1
    pieces = min(-(-3 * 304 // items), 256 // 64 + 1)
    assert pieces == 5
    rows = items * pieces * 128
    sched = _r256(16 + min(items * pieces, 304 * 2 + items) * 16 + items * 8)
    assert gqa.gqa_workspace_size(short, 256, 0) == _r256(sched + _r256(rows * 128 * 4) + rows * 4 * 4)


def test_workspace_plan_decode_large_group():
    # 16 query heads per KV head: one decode CTA per SM (its shared memory
    # does not fit twice), so 2 x 2 x 152 partial slots of 16 x (128 + 2)
    # floats, one arrival counter each and the chunk ticket
    d = dims(seq_len=1, head_size=128, num_heads=128, kv_num_heads=8, batch=4, max_seq_len=8192)
    slots = 2 * 2 * 152
    want = _r256(8 * (1 + slots)) + _r256(slots * 16 * 128 * 4) + _r256(slots * 16 * 2 * 4)
    assert gqa.gqa_workspace_size(d, 8192, 0) == want


def _header_text():
    text = open(os.path.join(ROOT, "include", "gqa.h")).read()
    return re.sub(r"/\*.*?\*/", "", text, flags=re.S)


def test_dims_struct_matches_header():
    """The ctypes mirror of gqa_dims_t has the header's fields, in order, all
    int32 (so the layout is the same on both sides)."""
    body = re.search(r"typedef struct \{(.*?)\}\s*gqa_dims_t;", _header_text(), flags=re.S).group(1)
    fields = re.findall(r"int32_t\s+(\w+)\s*;", body)
    assert [f for f, _ in gqa.gqa_dims_t._fields_] == fields
    assert all(t is ctypes.c_int32 for _, t in gqa.gqa_dims_t._fields_)
    assert ctypes.sizeof(gqa.gqa_dims_t) == 4 * len(fields)


def test_bound_argument_counts_match_header(lib):
    """Every function the binding declares takes as many arguments as the
    header's prototype."""
    text = _header_text()
    for name in gqa.EXPORTED:
        proto = re.search(r"\b" + name + r"\s*\((.*?)\)\s*;", text, flags=re.S).group(1)
        n = 0 if proto.strip() in ("", "void") else proto.count(",") + 1
        assert len(getattr(lib, name).argtypes) == n, name


def test_evicting_cache_host_rules(lib):
    """kv_eviction = 1: total_sequence_length beyond the buffer is no longer
    an overflow (the call goes on to the workspace check), the non-shared
    binding is not taken, and a call that may evict needs the evicting
    path's scratch (rotated queries and new key rows)."""
    d = dims(kv_eviction=1, cos_cache_rows=300)
    need = gqa.gqa_workspace_size(d, 300, 0)
    assert need >= (2 * 4 * 8 * 64 + 2 * 4 * 2 * 64) * 2
    assert need > gqa.gqa_workspace_size(d, 128, 0)     # a call that cannot evict takes the plain path
    assert call(d, total=300, workspace_bytes=need - 1) == gqa.GQA_ERR_INVALID_ARGUMENT
    assert call(dims(kv_eviction=1), total=300) == gqa.GQA_ERR_INVALID_ARGUMENT   # cos rows < total
    assert call(dims(cos_cache_rows=300), total=300) == gqa.GQA_ERR_KV_OVERFLOW
    ns = dict(present_key=0x200000, present_value=0x300000)
    assert call(dims(kv_eviction=1, past_seq_len=64), **ns) == gqa.GQA_ERR_UNSUPPORTED
    # the no-alloc entry does not take the evicting cache
    d1 = dims(kv_eviction=1, seq_len=1, head_size=128)
    st = gqa.gqa_decode_noalloc(d1, P["q"], P["k"], P["v"], P["kb"], P["vb"], P["kb"], P["vb"], P["seq"], 64,
                                P["cos"], P["sin"], 0.0, 0, None, P["out"], None)
    assert st == gqa.GQA_ERR_UNSUPPORTED
