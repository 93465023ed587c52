"""gqa_forward_host: the step with its per-call inputs (query, key, value,
seqlens_k) and its output in page-locked host memory, moved by the library's
copy kernels, checked against gqa_forward on the same inputs.  Both run the
same attention kernels on the same values, so outputs and buffers must agree
bit for bit.  Covered: the decode kernel, the tensor-core prefill with a bias
and key-range splits, and the generic path with a batch of 3 (a seqlens_k
copy that is not a multiple of 16 bytes, from an address that is only 4-byte
aligned).  Pointers that are not page-locked host memory are rejected before
any launch."""
import numpy as np
import pytest
import torch

import shared_kv_cache_gb300 as gqa
from shared_kv_cache_gb300 import workloads as W

from gqa_cases import run_cuda, to_device

GENERIC_B3 = W.Workload("host_generic_b3", "fp16", 3, 5, 8, 2, 64, 256, 0, 200, seed=61)


def _workload(name):
    return GENERIC_B3 if name == GENERIC_B3.name else W.CONFIGS[name]


def _dims(w, inp):
    bias = inp["attention_bias"]
    return gqa.make_dims(w.batch, w.seq_len, w.num_heads, w.kv_num_heads, w.head_size, w.max_seq_len, w.dtype, 0,
                         0 if inp["cos"] is None else inp["cos"].shape[0],
                         1 if bias is None else bias.shape[0], 1 if bias is None else bias.shape[1])


def _host_inputs(inp):
    hq = inp["query"].contiguous().pin_memory()
    hk = inp["key"].contiguous().pin_memory()
    hv = inp["value"].contiguous().pin_memory()
    # seqlens_k one int32 into a pinned buffer: 4-byte aligned, not 16
    sbuf = torch.zeros(inp["seqlens_k"].numel() + 1, dtype=torch.int32).pin_memory()
    sbuf[1:].copy_(inp["seqlens_k"])
    return hq, hk, hv, sbuf[1:]


def _call(w, inp, d, hq, hk, hv, hs, out, ws, stream):
    return gqa.gqa_forward_host(_dims(w, inp), hq, hk, hv, d["k_buf"], d["v_buf"], d["k_buf"], d["v_buf"], hs,
                                inp["total_sequence_length"], d["cos"], d["sin"], inp["scale"],
                                inp["local_window_size"], d["attention_bias"], out, ws, ws.numel(), stream)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["decode_b16", "chunked_prefill", GENERIC_B3.name])
def test_host_entry_matches_gqa_forward(name):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    w = _workload(name)
    inp = W.make_inputs(w)
    st, dst, ref_out, ref_kb, ref_vb = run_cuda(inp)
    assert st == gqa.GQA_OK and dst == gqa.GQA_OK, (gqa.gqa_status_string(st), gqa.gqa_status_string(dst))

    d = to_device(inp)
    hq, hk, hv, hs = _host_inputs(inp)
    nbytes = gqa.gqa_workspace_size_host(_dims(w, inp), inp["total_sequence_length"], inp["local_window_size"])
    assert nbytes >= gqa.gqa_workspace_size(_dims(w, inp), inp["total_sequence_length"], inp["local_window_size"])
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    # two calls in a row (the second one's copy-in follows the first one's
    # copy-out on the stream); each appends the same rows at the same slots
    outs = [torch.full(tuple(inp["query"].shape), float("nan"), dtype=inp["query"].dtype).pin_memory()
            for _ in range(2)]
    for out in outs:
        st = _call(w, inp, d, hq, hk, hv, hs, out, ws, stream)
        assert st == gqa.GQA_OK, gqa.gqa_status_string(st)
    dst = gqa.gqa_check_device_status(stream)  # synchronises the stream
    assert dst == gqa.GQA_OK, gqa.gqa_status_string(dst)
    for out in outs:
        assert np.array_equal(W.bits(out), W.bits(ref_out))
    assert np.array_equal(W.bits(d["k_buf"].cpu()), W.bits(ref_kb))
    assert np.array_equal(W.bits(d["v_buf"].cpu()), W.bits(ref_vb))


@pytest.mark.gpu
def test_host_entry_rejects_other_memory():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    w = GENERIC_B3
    inp = W.make_inputs(w)
    d = to_device(inp)
    hq, hk, hv, hs = _host_inputs(inp)
    out = torch.empty(tuple(inp["query"].shape), dtype=inp["query"].dtype).pin_memory()
    nbytes = gqa.gqa_workspace_size_host(_dims(w, inp), inp["total_sequence_length"], inp["local_window_size"])
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    kb0 = d["k_buf"].clone()
    stream = torch.cuda.current_stream()
    pageable = inp["query"].contiguous().clone()
    assert not pageable.is_pinned()
    for args in [(pageable, hk, hv, hs, out),            # pageable host memory
                 (d["query"], hk, hv, hs, out),          # device memory
                 (hq, hk, hv, hs, torch.empty_like(out, device="cpu", pin_memory=False))]:
        st = _call(w, inp, d, *args[:4], args[4], ws, stream)
        assert st == gqa.GQA_ERR_INVALID_ARGUMENT, gqa.gqa_status_string(st)
    assert gqa.gqa_check_device_status(stream) == gqa.GQA_OK
    # nothing was launched (bit compare: unused slots hold NaN sentinels)
    assert torch.equal(d["k_buf"].view(torch.int16), kb0.view(torch.int16))
