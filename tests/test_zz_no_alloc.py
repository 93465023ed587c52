"""gqa_decode_noalloc: the decode step for callers that cannot allocate device
memory when they run it (a runtime whose memory planner hands out every
buffer ahead of execution, a serving loop where cudaMalloc/cudaFree may not
synchronise the device).  Its scratch is a static 4 MiB device array inside
the library instead of a caller-supplied workspace.

The GPU tests call it through the C ABI, twice in a row, and check each
result against gqa_forward's on the same inputs (and the buffers bit for
bit), over the decode shapes of the parity tests: both element types, bias
shapes, group sizes 1 to 16, short and tile-edge lengths, windows, and a
sequence that overflows.  This file is collected last, so a run that stops at
the first failure has run every other test."""
import numpy as np
import pytest
import torch

import shared_kv_cache_gb300 as gqa
from shared_kv_cache_gb300 import workloads as W

from gqa_cases import TOL, custom, run_cuda, to_device

STATIC_SCRATCH_BYTES = 4 << 20


def static_partition_bytes(G, ctas):
    """Scratch of the static-partition decode kernels behind the entry point:
    two fp32 partials (G x 128 outputs, G (max, sum) pairs) per persistent
    CTA, whatever the lengths."""
    return ctas * 2 * G * (128 + 2) * 4 + 256


def _dims(inp):
    w = inp["workload"]
    bias = inp["attention_bias"]
    return gqa.make_dims(w.batch, w.seq_len, w.num_heads, w.kv_num_heads, w.head_size, w.max_seq_len, w.dtype,
                         inp.get("rotary_interleaved", 0), 0 if inp["cos"] is None else inp["cos"].shape[0],
                         1 if bias is None else bias.shape[0], 1 if bias is None else bias.shape[1])


def _noalloc(inp, d, stream):
    """One gqa_decode_noalloc call on device inputs d; returns (status,
    device status, output on the CPU)."""
    w = inp["workload"]
    out = torch.full_like(d["query"], float("nan"))
    st = gqa.gqa_decode_noalloc(_dims(inp), d["query"], d["key"], d["value"], d["k_buf"], d["v_buf"], d["k_buf"],
                                d["v_buf"], d["seqlens_k"], inp["total_sequence_length"], d["cos"], d["sin"],
                                inp["scale"], w.local_window_size, d["attention_bias"], out, stream)
    return st, gqa.gqa_check_device_status(stream), out.cpu()


CASES = {
    "decode_b16": lambda: W.make_inputs(W.CONFIGS["decode_b16"]),
    "long_decode_w4096": lambda: W.make_inputs(W.CONFIGS["long_decode_w4096"]),
    "fp16": lambda: custom(dtype="fp16", seed=201),
    "bias_1x1": lambda: custom(bias=(1, 1), seed=202),
    "bias_BxH_fp16": lambda: custom(bias=(3, 8), dtype="fp16", seed=203),
    "group16": lambda: custom(H=16, Hkv=1, seed=204),
    "group1": lambda: custom(H=4, Hkv=4, seed=205),
    "short_and_tile_edges": lambda: custom(past=(0, 1, 63, 64, 65, 127, 128, 999), B=8, seed=206),
    "interleaved_window": lambda: custom(interleaved=1, window=100, seed=207),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_gqa_forward_on_two_calls(name):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    inp = CASES[name]()
    w = inp["workload"]
    # the existing entry point, with a workspace, on its own copy of the inputs
    st, dst, ref_out, ref_kb, ref_vb = run_cuda(inp)
    assert st == gqa.GQA_OK and dst == gqa.GQA_OK
    ref = ref_out.double().numpy()

    d = to_device(inp)
    stream = torch.cuda.current_stream()
    # another shape (larger batch and group) in between leaves other partials
    # in the shared array: the next call must not depend on them
    other = custom(B=6, H=16, Hkv=2, M=700, past=(699, 0, 345, 12, 640, 64), seed=208)
    od = to_device(other)
    for k in range(2):
        st, dst, out = _noalloc(inp, d, stream)
        assert st == gqa.GQA_OK, gqa.gqa_status_string(st)
        assert dst == gqa.GQA_OK, gqa.gqa_status_string(dst)
        got = out.double().numpy()
        assert np.all(np.isfinite(got))
        assert np.abs(got - ref).max() <= TOL[w.dtype]
        assert np.array_equal(W.bits(d["k_buf"].cpu()), W.bits(ref_kb))
        assert np.array_equal(W.bits(d["v_buf"].cpu()), W.bits(ref_vb))
        if k == 0:
            st, dst, _ = _noalloc(other, od, stream)
            assert st == gqa.GQA_OK and dst == gqa.GQA_OK


@pytest.mark.gpu
def test_noalloc_device_overflow_matches_gqa_forward():
    """A sequence whose past length leaves no room: GQA_ERR_KV_OVERFLOW from
    gqa_check_device_status, that sequence skipped, the others computed as
    gqa_forward computes them."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    inp = custom(M=600, past=(10, 600, 300), total=600, seed=209)
    st, dst, ref_out, ref_kb, ref_vb = run_cuda(inp)
    assert st == gqa.GQA_OK and dst == gqa.GQA_ERR_KV_OVERFLOW
    d = to_device(inp)
    stream = torch.cuda.current_stream()
    st, dst, out = _noalloc(inp, d, stream)
    assert st == gqa.GQA_OK and dst == gqa.GQA_ERR_KV_OVERFLOW
    assert torch.isnan(out[1].float()).all()
    assert np.abs(out[[0, 2]].double().numpy() - ref_out[[0, 2]].double().numpy()).max() <= TOL["bf16"]
    assert np.array_equal(W.bits(d["k_buf"].cpu()), W.bits(ref_kb))
    assert np.array_equal(W.bits(d["v_buf"].cpu()), W.bits(ref_vb))


@pytest.mark.gpu
def test_noalloc_scratch_fits_on_this_device():
    """The bound computed from this device's SM count (two resident CTAs per
    SM up to 8 query heads per KV head, one above), and every group size
    accepted by the entry point here."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for G in (1, 4, 8, 16):
        assert static_partition_bytes(G, (2 if G <= 8 else 1) * sms) <= STATIC_SCRATCH_BYTES
        inp = custom(H=G, Hkv=1, B=2, past=(5, 300), M=400, seed=210 + G)
        st, dst, out = _noalloc(inp, to_device(inp), torch.cuda.current_stream())
        assert st == gqa.GQA_OK and dst == gqa.GQA_OK, (G, gqa.gqa_status_string(st))


def test_noalloc_scratch_bound_and_rejected_shapes():
    """The static-partition decode kernels need at most two partials of
    G x (128 + 2) floats per persistent CTA, whatever the lengths, so every
    decode shape fits the static array on a 152-SM GB300; shapes other than
    the decode shape are rejected before any launch (the pointers below are
    never dereferenced)."""
    gqa.load_library()
    for G in (1, 4, 8, 16):
        assert static_partition_bytes(G, (2 if G <= 8 else 1) * 152) <= STATIC_SCRATCH_BYTES
    p = [0x100000 * (i + 1) for i in range(12)]
    d2 = gqa.make_dims(2, 4, 8, 2, 128, 256, "fp16", 0, 256, 1, 1)   # four new tokens: not a decode step
    st = gqa.gqa_decode_noalloc(d2, p[0], p[1], p[2], p[3], p[4], p[3], p[4], p[5], 64, p[6], p[7], 0.0, 0,
                                None, p[8], None)
    assert st == gqa.GQA_ERR_UNSUPPORTED
    d3 = gqa.make_dims(2, 1, 8, 2, 64, 256, "fp16", 0, 256, 1, 1)    # head size 64
    st = gqa.gqa_decode_noalloc(d3, p[0], p[1], p[2], p[3], p[4], p[3], p[4], p[5], 64, p[6], p[7], 0.0, 0,
                                None, p[8], None)
    assert st == gqa.GQA_ERR_UNSUPPORTED
