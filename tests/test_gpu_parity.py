"""CUDA path versus the CPU oracle, through the C ABI, on seeded inputs.

KV append: bit-exact over the whole buffer (slots outside the new tokens keep
their NaN sentinel or past values).  Attention output: max-abs error within
2e-3 (fp16) / 1e-2 (bf16) of the oracle's float64 result."""
import numpy as np
import pytest
import torch

import oracle
import shared_kv_cache_gb300 as gqa
from shared_kv_cache_gb300 import workloads as W

from gqa_cases import compare, custom, run_cuda, run_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    gqa.load_library()


def check(inp, heads=None, batches=None):
    res = run_cuda(inp)
    ref = run_oracle(inp, heads=heads, batches=batches)
    return compare(inp, res, ref, heads=heads, batches=batches)


# ---------------------------------------------------------------------------
# The five workloads at their full sizes
# ---------------------------------------------------------------------------
def test_tiny_prefill_then_decode():
    """32-token prompt (head size 8) into an empty past, then one decode token
    over the grown sequence of 33."""
    w = W.CONFIGS["tiny_prefill"]
    inp = W.make_inputs(w)
    res = run_cuda(inp)
    ref = run_oracle(inp)
    compare(inp, res, ref)
    wd = W.CONFIGS["tiny_decode"]
    dec = W.make_inputs(wd, seed=1)
    dec["k_buf"] = res[3].clone()
    dec["v_buf"] = res[4].clone()
    dec["seqlens_k"] = torch.tensor([32], dtype=torch.int32)
    dec["total_sequence_length"] = 33
    compare(dec, run_cuda(dec), run_oracle(dec))


def test_decode_b16_full():
    check(W.make_inputs(W.CONFIGS["decode_b16"]))


def test_prefill_2k_full():
    """Every head of every sequence (4 x 2048 rows x 32 heads)."""
    check(W.make_inputs(W.CONFIGS["prefill_2k"]))


def test_chunked_prefill_full_with_bias():
    check(W.make_inputs(W.CONFIGS["chunked_prefill"]))


@pytest.mark.parametrize("name", ["long_decode", "long_decode_w4096"])
def test_long_decode_full(name):
    """All 64 heads of all 8 sequences."""
    check(W.make_inputs(W.CONFIGS[name]))


def test_chunked_overflow_is_an_error_and_writes_nothing():
    w = W.CONFIGS["chunked_overflow"]
    inp = W.make_inputs(w)
    kb0, vb0 = W.bits(inp["k_buf"]).copy(), W.bits(inp["v_buf"]).copy()
    # host-visible: total_sequence_length = past + new = 4128 > max_seq_len
    st, dst, out, kb, vb = run_cuda(inp, total=4128)
    assert st == gqa.GQA_ERR_KV_OVERFLOW and dst == gqa.GQA_OK
    assert np.array_equal(W.bits(kb), kb0) and np.array_equal(W.bits(vb), vb0)
    # device-visible: the host is told total = 4096, seqlens_k says 4000 + 128
    st, dst, out, kb, vb = run_cuda(inp)
    assert st == gqa.GQA_OK and dst == gqa.GQA_ERR_KV_OVERFLOW
    assert np.array_equal(W.bits(kb), kb0) and np.array_equal(W.bits(vb), vb0)
    assert torch.isnan(out.float()).all()   # no output row written for the skipped sequence
    assert run_oracle(inp, total_sequence_length=4128)[0] == oracle.STATUS_KV_OVERFLOW


# ---------------------------------------------------------------------------
# Decode path: ragged lengths, tails, windows, bias, group sizes
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("kw", [
    dict(),
    dict(dtype="fp16"),
    dict(past=(0, 1, 63, 64, 65, 127, 128, 999), B=8, seed=8),
    dict(H=16, Hkv=1, seed=9),                      # G = 16
    dict(H=4, Hkv=4, seed=10),                      # G = 1 (MHA)
    dict(H=12, Hkv=4, seed=11),                     # G = 3
    dict(window=100, seed=12),
    dict(window=1, seed=13),
    dict(window=64, past=(63, 64, 200), seed=14),
    dict(bias=(1, 1), seed=15),
    dict(bias=(3, 8), dtype="fp16", seed=16),
    dict(rotary=False, seed=17),
    dict(interleaved=1, seed=18),
    dict(M=4096, past=(4095, 3000, 17), total=4096, seed=19),   # the last slot of the buffer
    # many short items and a few long ones: CTAs see many segments each
    dict(B=40, H=16, Hkv=4, M=3000, past=tuple([0, 1, 2, 63, 64, 65] * 6 + [2999, 1500, 777, 128]), seed=22),
    dict(B=40, H=16, Hkv=4, M=3000, past=tuple([5] * 39 + [2999]), window=700, seed=23),
])
def test_decode_cases(kw):
    check(custom(**kw))


def test_decode_device_overflow_skips_that_sequence():
    inp = custom(M=600, past=(10, 600, 300), total=600, seed=20)
    kb0, vb0 = W.bits(inp["k_buf"]).copy(), W.bits(inp["v_buf"]).copy()
    st, dst, out, kb, vb = run_cuda(inp)
    assert st == gqa.GQA_OK and dst == gqa.GQA_ERR_KV_OVERFLOW
    assert np.array_equal(W.bits(kb)[1], kb0[1]) and np.array_equal(W.bits(vb)[1], vb0[1])
    assert torch.isnan(out[1].float()).all()
    # the other sequences are computed as usual
    ok = custom(M=600, past=(10, 300), total=600, seed=20, B=2)
    ok["query"], ok["key"], ok["value"] = (inp[n][[0, 2]].contiguous() for n in ("query", "key", "value"))
    ok["k_buf"], ok["v_buf"] = inp["k_buf"][[0, 2]].contiguous(), inp["v_buf"][[0, 2]].contiguous()
    ref = run_oracle(ok)
    assert np.array_equal(W.bits(kb)[[0, 2]], ref[2]) and np.array_equal(W.bits(vb)[[0, 2]], ref[3])
    got = out[[0, 2]].double().numpy()
    assert np.abs(got - ref[1]).max() <= 1e-2


def test_decode_repeat_is_idempotent():
    inp = custom(seed=21)
    a = run_cuda(inp)
    b = run_cuda(inp)
    assert all(np.array_equal(W.bits(x), W.bits(y)) for x, y in zip(a[2:], b[2:]))


# ---------------------------------------------------------------------------
# Prefill / generic path
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("kw", [
    dict(S=37, past=(0, 5, 90), M=160, dtype="fp16", seed=30),
    dict(S=37, past=(0, 5, 90), M=160, dtype="bf16", bias=(3, 8), seed=31),
    dict(S=130, past=(0, 129, 7), M=300, window=50, seed=32),
    dict(S=5, D=64, past=(3, 0, 40), M=64, seed=33),
    dict(S=5, D=256, past=(3, 0, 40), M=64, seed=34),
    dict(S=9, D=24, H=6, Hkv=3, past=(1, 2, 3), M=16, seed=35),
    dict(S=1, D=64, past=(3, 0, 40), M=64, seed=36),
    dict(S=16, D=8, H=4, Hkv=2, past=(0, 4, 8), M=32, interleaved=1, seed=37),
    dict(S=16, D=128, rotary=False, past=(0, 4, 8), M=32, seed=38),
    # tensor-core prefill: several query and key tiles, ragged tails, bias paths, windows
    dict(S=200, past=(0, 77, 1000), M=1304, total=1304, dtype="bf16", bias=(1, 1), seed=40),
    dict(S=200, past=(3, 77, 1001), M=1300, total=1300, dtype="fp16", bias=(3, 8), seed=41),
    dict(S=129, past=(5, 0, 300), M=512, window=100, bias=(3, 1), seed=42),
    dict(S=257, past=(0, 130, 255), M=600, window=300, dtype="bf16", seed=43),
    dict(S=128, past=(128, 0, 383), M=512, H=16, Hkv=2, seed=44),
    # query rotation inside the tensor-core kernel: interleaved pairs, and an
    # odd group size (the last head of each KV head runs alone)
    dict(S=150, past=(0, 40, 300), M=512, interleaved=1, seed=45),
    dict(S=140, past=(2, 0, 200), M=400, H=12, Hkv=4, interleaved=1, dtype="bf16", seed=46),
    dict(S=70, past=(9, 0, 31), M=128, H=6, Hkv=2, seed=47),
])
def test_prefill_cases(kw):
    check(custom(**kw))


# ---------------------------------------------------------------------------
# Tensor-core prefill grids of at least two CTAs per CTA slot (B x H x
# 128-token query tiles >= 2 x 2 x SMs): one CTA per work item, no work list
# and no split key ranges (the cases above take the list)
# ---------------------------------------------------------------------------
def _full_grid(inp):
    w = inp["workload"]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    items = w.batch * w.num_heads * -(-w.seq_len // 128)
    if items < 4 * sms:
        pytest.skip(f"{items} work items do not fill two CTAs per slot on {sms} SMs")
    # no work list, no partials: no scratch
    dims = gqa.make_dims(w.batch, w.seq_len, w.num_heads, w.kv_num_heads, w.head_size, w.max_seq_len, w.dtype, 0,
                         0 if inp["cos"] is None else inp["cos"].shape[0])
    assert gqa.gqa_workspace_size(dims, inp["total_sequence_length"], inp["local_window_size"]) == 0


@pytest.mark.parametrize("kw", [
    # ragged pasts around 64-key tiles; G = 10
    dict(S=160, B=4, H=80, Hkv=8, past=(0, 37, 300, 1000), M=1200, dtype="fp16", seed=90),
    # window, bias, interleaved rotary, bf16; G = 13
    dict(S=300, B=2, H=104, Hkv=8, past=(5, 700), M=1100, window=100, bias=(1, 1), interleaved=1, dtype="bf16",
         seed=91),
    # no rotary; pasts at and next to tile edges
    dict(S=129, B=5, H=64, Hkv=4, past=(0, 1, 63, 64, 65), M=256, rotary=False, dtype="fp16", seed=92),
    # the two-head kernel (even group size, no window, no bias): bf16 rows
    # that see few keys (P's residue), interleaved rotary; G = 20
    dict(S=256, B=2, H=160, Hkv=8, past=(0, 100), M=512, interleaved=1, dtype="bf16", seed=94),
    # ragged query tiles (S = 300) and 128-key tiles straddling the past; G = 26
    dict(S=300, B=2, H=104, Hkv=4, past=(5, 700), M=1100, dtype="fp16", seed=95),
])
def test_full_grid_prefill_cases(kw):
    inp = custom(**kw)
    _full_grid(inp)
    check(inp)


@pytest.mark.parametrize("H", [152, 160])  # group sizes 19 (one head per CTA) and 20 (two)
def test_full_grid_prefill_device_overflow_skips_that_sequence(H):
    """One sequence's past + new exceeds max_seq_len (the host is told a
    total that fits): the error word says so, that sequence's buffer rows and
    output rows are untouched, and the others match the oracle."""
    kw = dict(S=128, B=4, H=H, Hkv=8, M=4096, total=4096, dtype="fp16", seed=93)
    inp = custom(past=(0, 3969, 100, 3968), **kw)
    _full_grid(inp)
    kb0, vb0 = W.bits(inp["k_buf"]).copy(), W.bits(inp["v_buf"]).copy()
    st, dst, out, kb, vb = run_cuda(inp)
    assert st == gqa.GQA_OK and dst == gqa.GQA_ERR_KV_OVERFLOW
    assert np.array_equal(W.bits(kb)[1], kb0[1]) and np.array_equal(W.bits(vb)[1], vb0[1])
    assert torch.isnan(out[1].float()).all()
    keep = [0, 2, 3]
    ok = custom(past=(0, 100, 3968), **{**kw, "B": 3})
    for n in ("query", "key", "value", "k_buf", "v_buf"):
        ok[n] = inp[n][keep].contiguous()
    ref = run_oracle(ok)
    assert np.array_equal(W.bits(kb)[keep], ref[2]) and np.array_equal(W.bits(vb)[keep], ref[3])
    got = out[keep].double().numpy()
    assert np.abs(got - ref[1].reshape(got.shape)).max() <= 2e-3


# ---------------------------------------------------------------------------
# Non-shared binding: separate past [B, Hkv, Mp, D] and present buffers; the
# present becomes past + new
# ---------------------------------------------------------------------------
def _split(inp, Mp, seed):
    """Moves the case's past rows into separate past buffers of Mp slots
    (later slots random: not part of the past) and makes the present buffers
    all sentinel."""
    w = inp["workload"]
    gen = torch.Generator().manual_seed(seed)
    past = {}
    for name in ("k_buf", "v_buf"):
        pk = torch.randn(w.batch, w.kv_num_heads, Mp, w.head_size, generator=gen).to(W.DTYPES[w.dtype])
        for b, n in enumerate(inp["seqlens_k"].tolist()):
            pk[b, :, :min(n, Mp)] = inp[name][b, :, :min(n, Mp)]
        past[name] = pk
        fresh = torch.empty(inp[name].shape, dtype=torch.int16).fill_(W.SENTINEL_BITS[w.dtype])
        inp[name] = fresh.view(W.DTYPES[w.dtype])
    return past


def _run_cuda_split(inp, past):
    w = inp["workload"]
    d = to_device(inp)
    pk, pv = past["k_buf"].cuda(), past["v_buf"].cuda()
    out = torch.full_like(d["query"], float("nan"))
    bias = d["attention_bias"]
    dims = gqa.make_dims(w.batch, w.seq_len, w.num_heads, w.kv_num_heads, w.head_size, w.max_seq_len, w.dtype, 0,
                         d["cos"].shape[0], 1 if bias is None else bias.shape[0],
                         1 if bias is None else bias.shape[1], past_seq_len=pk.shape[2])
    total = inp["total_sequence_length"]
    ws = torch.empty(max(gqa.gqa_workspace_size(dims, total, inp["local_window_size"]), 256), dtype=torch.uint8,
                     device="cuda")
    st = gqa.gqa_forward(dims, d["query"], d["key"], d["value"], pk, pv, d["k_buf"], d["v_buf"], d["seqlens_k"],
                         total, d["cos"], d["sin"], inp["scale"], inp["local_window_size"], bias, out, ws,
                         ws.numel(), None)
    dst = gqa.gqa_check_device_status(None)
    return (st, dst, out.cpu(), d["k_buf"].cpu(), d["v_buf"].cpu()), (pk.cpu(), pv.cpu())


@pytest.mark.parametrize("kw", [
    dict(dtype="bf16", B=3, S=1, H=8, Hkv=2, D=128, M=1000, past=(0, 517, 999), seed=81),   # decode kernel
    dict(dtype="fp16", B=2, S=64, H=8, Hkv=2, D=128, M=512, past=(0, 300), bias=(1, 1), seed=82),  # tcgen05 prefill
    dict(dtype="fp16", B=3, S=5, H=8, Hkv=2, D=64, M=256, past=(0, 17, 200), seed=83),      # generic path
])
def test_non_shared_binding(kw):
    """The present buffers come back as past + new (bit for bit), the past
    buffers unchanged, and the output matches the oracle."""
    inp = custom(**kw)
    Mp = min(kw["M"], max(kw["past"]) + 7)
    past = _split(inp, Mp, seed=kw["seed"] + 500)
    past_bits = {n: W.bits(t).copy() for n, t in past.items()}
    res, (pk, pv) = _run_cuda_split(inp, past)
    ref = run_oracle(inp, past_key=past_bits["k_buf"], past_value=past_bits["v_buf"])
    compare(inp, res, ref)
    assert np.array_equal(W.bits(pk), past_bits["k_buf"]) and np.array_equal(W.bits(pv), past_bits["v_buf"])


def test_non_shared_past_shorter_than_a_length_records_an_error():
    """A sequence whose past length is beyond the past's Mp slots records
    GQA_ERR_INVALID_ARGUMENT and its present slots below that length are not
    copied; the past is not written."""
    inp = custom(dtype="bf16", B=3, S=1, H=8, Hkv=2, D=128, M=1000, past=(0, 517, 999), seed=84)
    past = _split(inp, 600, seed=584)
    past_bits = {n: W.bits(t).copy() for n, t in past.items()}
    (st, dst, _, kb, vb), (pk, pv) = _run_cuda_split(inp, past)
    assert st == gqa.GQA_OK and dst == gqa.GQA_ERR_INVALID_ARGUMENT
    sentinel = W.SENTINEL_BITS["bf16"]
    assert np.all(W.bits(kb)[2, :, :999] == sentinel) and np.all(W.bits(vb)[2, :, :999] == sentinel)
    assert np.array_equal(W.bits(kb)[1, :, :517], past_bits["k_buf"][1, :, :517])
    assert np.array_equal(W.bits(pk), past_bits["k_buf"]) and np.array_equal(W.bits(pv), past_bits["v_buf"])
