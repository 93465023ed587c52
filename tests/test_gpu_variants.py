"""GPU parity of the operator variants against the CPU oracle, through the C
ABI: packed QKV input (one query tensor holding each token's query, key and
value heads) and the sliding-window cache with contiguous eviction
(dims.kv_eviction = 1).  The buffers are compared bit for bit in full, the
outputs within the dtype's tolerance."""
import numpy as np
import pytest
import torch

import oracle
import shared_kv_cache_gb300 as gqa
from shared_kv_cache_gb300 import workloads as W

from gqa_cases import compare, custom, dims_of, pack_qkv, run_cuda, run_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    gqa.load_library()


# ---------------------------------------------------------------------------
# Packed QKV
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("kw", [
    dict(seed=301),                                                   # decode kernel
    dict(dtype="fp16", H=16, Hkv=1, window=100, seed=302),            # decode, G = 16, window
    dict(S=200, past=(0, 77, 1000), M=1304, total=1304, bias=(1, 1), seed=303),    # tensor-core prefill
    dict(S=150, past=(0, 40, 300), M=512, interleaved=1, dtype="fp16", seed=304),  # prefill, interleaved
    dict(S=5, D=64, past=(3, 0, 40), M=64, seed=305),                 # generic kernel
    dict(S=4, D=128, rotary=False, past=(0, 4, 8), M=32, seed=306),   # prefill without rotary
    # a grid of 640 one-head items (the two-head prefill kernel on 152 SMs),
    # G = 20, ragged pasts, interleaved rotary
    dict(S=128, B=4, H=160, Hkv=8, past=(0, 50, 130, 7), M=512, interleaved=1, seed=307),
])
def test_packed_qkv_matches_oracle(kw):
    inp = custom(**kw)
    res = run_cuda(inp, packed=True)
    packed = W.bits(pack_qkv(inp))
    ref = run_oracle(inp, query=packed, key=None, value=None)
    compare(inp, res, ref)


def test_packed_qkv_host_buffer_entry():
    """gqa_forward_host with the packed rows in pinned host memory gives the
    device entry's bits."""
    inp = custom(seed=307)
    st, dst, ref_out, ref_kb, ref_vb = run_cuda(inp, packed=True)
    assert st == gqa.GQA_OK and dst == gqa.GQA_OK
    w = inp["workload"]
    d = to_device(inp)
    hq = pack_qkv(inp).pin_memory()
    hs = inp["seqlens_k"].clone().pin_memory()
    stream = torch.cuda.current_stream()
    out = gqa.forward_host(hq, None, None, d["k_buf"], d["v_buf"], hs, inp["total_sequence_length"],
                           w.num_heads, w.kv_num_heads, d["cos"], d["sin"], inp["scale"], 0, None, stream=stream)
    stream.synchronize()
    assert gqa.gqa_check_device_status(stream) == gqa.GQA_OK
    assert np.array_equal(W.bits(out), W.bits(ref_out))
    assert np.array_equal(W.bits(d["k_buf"].cpu()), W.bits(ref_kb))


def test_one_of_key_value_missing_is_invalid():
    inp = custom(seed=308)
    d = to_device(inp)
    dims = dims_of(inp)
    out = torch.empty_like(d["query"])
    ws = torch.empty(max(gqa.gqa_workspace_size(dims, inp["total_sequence_length"], 0), 256), dtype=torch.uint8,
                     device="cuda")
    st = gqa.gqa_forward(dims, d["query"], d["key"], None, d["k_buf"], d["v_buf"], d["k_buf"], d["v_buf"],
                         d["seqlens_k"], inp["total_sequence_length"], d["cos"], d["sin"], 0.0, 0, None, out, ws,
                         ws.numel(), None)
    assert st == gqa.GQA_ERR_INVALID_ARGUMENT


# ---------------------------------------------------------------------------
# Sliding-window cache with contiguous eviction
# ---------------------------------------------------------------------------
EVICT_CASES = [
    # decode kernel: empty, partial, exactly full, full, long past the capacity
    dict(B=5, M=300, past=(0, 150, 299, 300, 1000), seed=401),
    dict(B=5, M=300, past=(0, 150, 299, 300, 1000), window=100, dtype="fp16", seed=402),
    dict(B=5, M=300, past=(7, 299, 300, 301, 5000), window=300, seed=403),
    dict(B=4, M=256, past=(255, 256, 257, 700), H=16, Hkv=1, bias=(1, 1), seed=404),
    dict(B=3, M=200, past=(199, 400, 64), H=4, Hkv=4, interleaved=1, bias=(3, 4), seed=405),
    dict(B=3, M=128, past=(127, 128, 129), rotary=False, seed=406),
    # generic kernel: several new tokens, other head sizes
    dict(B=4, S=5, M=64, past=(0, 60, 64, 200), seed=407),
    dict(B=4, S=5, M=64, past=(0, 60, 64, 200), window=20, dtype="fp16", bias=(1, 8), seed=408),
    dict(B=3, S=70, M=64, past=(0, 10, 100), seed=409),            # more new tokens than the capacity
    dict(B=3, S=1, D=64, M=50, past=(49, 50, 123), window=10, seed=410),
    dict(B=2, S=3, D=8, H=4, Hkv=2, M=16, past=(15, 40), interleaved=1, dtype="fp16", seed=411),
]


@pytest.mark.parametrize("kw", EVICT_CASES)
def test_evicting_cache_matches_oracle(kw):
    inp = custom(evict=True, **kw)
    assert inp["total_sequence_length"] > inp["workload"].max_seq_len  # the call may evict
    compare(inp, run_cuda(inp), run_oracle(inp))


@pytest.mark.parametrize("dtype,window", [("bf16", 0), ("fp16", 96)])
def test_evicting_decode_loop(dtype, window):
    """Twelve decode steps into a cache of 128 slots that fills and then
    evicts every step: the buffer carried on the GPU matches the oracle's
    buffer bit for bit after every step, and every output row matches."""
    B, H, Hkv, D, M = 3, 8, 2, 128, 128
    start = [120, 128, 300]
    inp = custom(dtype=dtype, B=B, H=H, Hkv=Hkv, D=D, M=M, past=start, window=window, evict=True, seed=420,
                 total=max(start) + 12)
    kb_gpu, vb_gpu = inp["k_buf"].cuda(), inp["v_buf"].cuda()
    kb_ref, vb_ref = W.bits(inp["k_buf"]).copy(), W.bits(inp["v_buf"]).copy()
    gen = torch.Generator().manual_seed(421)
    dims = dims_of(inp)
    total = inp["total_sequence_length"]
    ws = torch.empty(max(gqa.gqa_workspace_size(dims, total, window), 256), dtype=torch.uint8, device="cuda")
    cos, sin = inp["cos"].cuda(), inp["sin"].cuda()
    t = W.DTYPES[dtype]
    for step in range(12):
        past = torch.tensor([p + step for p in start], dtype=torch.int32)
        q = torch.randn(B, 1, H * D, generator=gen).to(t)
        k = torch.randn(B, 1, Hkv * D, generator=gen).to(t)
        v = torch.randn(B, 1, Hkv * D, generator=gen).to(t)
        out = torch.full((B, 1, H * D), float("nan"), dtype=t, device="cuda")
        st = gqa.gqa_forward(dims, q.cuda(), k.cuda(), v.cuda(), kb_gpu, vb_gpu, kb_gpu, vb_gpu, past.cuda(), total,
                             cos, sin, inp["scale"], window, None, out, ws, ws.numel(), None)
        assert st == gqa.GQA_OK and gqa.gqa_check_device_status(None) == gqa.GQA_OK
        ost, oout, kb_ref, vb_ref = oracle.gqa_forward(
            W.bits(q), W.bits(k), W.bits(v), kb_ref, vb_ref, past.numpy(), total, W.bits(inp["cos"]),
            W.bits(inp["sin"]), H, Hkv, inp["scale"], window, None, dtype, evict=True)
        assert ost == oracle.STATUS_OK
        assert np.array_equal(W.bits(kb_gpu.cpu()), kb_ref), step
        assert np.array_equal(W.bits(vb_gpu.cpu()), vb_ref), step
        err = np.abs(out.cpu().double().numpy() - oout).max()
        assert err <= {"fp16": 2e-3, "bf16": 1e-2}[dtype], (step, err)


def test_evicting_mode_without_overflow_uses_the_plain_path():
    """kv_eviction = 1 with total_sequence_length <= M: no sequence can
    evict, the result is the plain append's; a sequence beyond
    total_sequence_length is an invalid argument (not an overflow)."""
    inp = custom(M=1000, past=(0, 517, 990), evict=True, seed=430)
    compare(inp, run_cuda(inp), run_oracle(inp))
    bad = custom(M=600, past=(10, 599, 300), total=600, evict=True, seed=431)
    bad["seqlens_k"] = torch.tensor([10, 600, 300], dtype=torch.int32)   # 600 + 1 > total
    st, dst, out, kb, vb = run_cuda(bad)
    assert st == gqa.GQA_OK and dst == gqa.GQA_ERR_INVALID_ARGUMENT
    assert torch.isnan(out[1].float()).all()


# ---------------------------------------------------------------------------
# Determinism of the split prefill
# ---------------------------------------------------------------------------
def test_split_prefill_gives_the_same_bits_every_call():
    """The chunked prefill's items are cut into pieces whose partials the
    item's last piece merges; which piece is last varies from call to call,
    the merged output must not."""
    inp = W.make_inputs(W.CONFIGS["chunked_prefill"])
    outs = [W.bits(run_cuda(inp)[2]) for _ in range(4)]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
