"""gqa_decode_noalloc: the decode step for callers that cannot allocate device
memory when they run it (a runtime whose memory planner hands out every
buffer ahead of execution, a serving loop where cudaMalloc/cudaFree may not
synchronise the device).  Its scratch is a static 4 MiB device array inside
the library instead of a caller-supplied workspace.

The GPU test calls it twice in a row through the C ABI and checks each
result against gqa_forward's on the same inputs.  This file is collected
last, so a run that stops at the first failure has run every other test."""
import numpy as np
import pytest
import torch

import shared_kv_cache_gb300 as gqa
from shared_kv_cache_gb300 import workloads as W

from gqa_cases import TOL, run_cuda, to_device

STATIC_SCRATCH_BYTES = 4 << 20


def static_partition_bytes(G, ctas):
    """Scratch of the static-partition decode kernels behind the entry point:
    two fp32 partials (G x 128 outputs, G (max, sum) pairs) per persistent
    CTA, whatever the lengths."""
    return ctas * 2 * G * (128 + 2) * 4 + 256


def _dims(w, inp):
    return gqa.make_dims(w.batch, w.seq_len, w.num_heads, w.kv_num_heads, w.head_size, w.max_seq_len, w.dtype,
                         0, inp["cos"].shape[0], 1, 1)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["decode_b16", "long_decode_w4096"])
def test_noalloc_matches_gqa_forward_on_two_calls(name):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    w = W.CONFIGS[name]
    inp = W.make_inputs(w)
    dims = _dims(w, inp)
    assert static_partition_bytes(w.group, 2 * 152) <= STATIC_SCRATCH_BYTES
    # the existing entry point, with a workspace, on its own copy of the inputs
    st, dst, ref_out, ref_kb, ref_vb = run_cuda(inp)
    assert st == gqa.GQA_OK and dst == gqa.GQA_OK
    ref = ref_out.double().numpy()

    d = to_device(inp)
    stream = torch.cuda.current_stream()
    for _ in range(2):
        out = torch.full_like(d["query"], float("nan"))
        st = gqa.gqa_decode_noalloc(dims, d["query"], d["key"], d["value"], d["k_buf"], d["v_buf"], d["k_buf"],
                                    d["v_buf"], d["seqlens_k"], inp["total_sequence_length"], d["cos"], d["sin"],
                                    inp["scale"], w.local_window_size, None, out, stream)
        assert st == gqa.GQA_OK, gqa.gqa_status_string(st)
        dst = gqa.gqa_check_device_status(stream)
        assert dst == gqa.GQA_OK, gqa.gqa_status_string(dst)
        got = out.cpu().double().numpy()
        assert np.all(np.isfinite(got))
        assert np.abs(got - ref).max() <= TOL[w.dtype]
        assert np.array_equal(W.bits(d["k_buf"].cpu()), W.bits(ref_kb))
        assert np.array_equal(W.bits(d["v_buf"].cpu()), W.bits(ref_vb))


def test_noalloc_scratch_bound_and_rejected_shapes():
    """The static-partition decode kernels need at most two partials of
    G x (128 + 2) floats per persistent CTA, whatever the lengths (two CTAs
    per SM up to 8 heads per KV head, one above, on 152 SMs), so every decode
    shape fits the static array; shapes other than the decode shape are
    rejected before any launch (the pointers below are never dereferenced)."""
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
