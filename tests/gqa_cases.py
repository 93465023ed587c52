"""Shared helpers for the tests: run one GroupQueryAttention call through the
C ABI on the GPU, and the same inputs through the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import shared_kv_cache_gb300 as gqa
from shared_kv_cache_gb300 import workloads as W

# Attention output tolerance (max abs against the oracle's float64 result):
# 2e-3 for fp16, 1e-2 for bf16, but never finer than one unit in the last
# place of the output type at the reference value -- an output stored in T
# cannot resolve more than that (for |o| >= 2 in bf16, >= 4 in fp16).
TOL = {"fp16": 2e-3, "bf16": 1e-2}


def to_device(inp: dict, device="cuda") -> dict:
    out = {}
    for k, v in inp.items():
        out[k] = v.to(device) if isinstance(v, torch.Tensor) else v
    return out


def run_cuda(inp: dict, stream=None, total=None, workspace_pad=0):
    """Returns (status, device_status, out[CPU], k_buf[CPU], v_buf[CPU])."""
    w = inp["workload"]
    d = to_device(inp)
    out = torch.full_like(d["query"], float("nan"))
    dims = gqa.make_dims(w.batch, w.seq_len, w.num_heads, w.kv_num_heads, w.head_size, w.max_seq_len, w.dtype,
                         inp.get("rotary_interleaved", 0),
                         0 if d["cos"] is None else d["cos"].shape[0],
                         1 if d["attention_bias"] is None else d["attention_bias"].shape[0],
                         1 if d["attention_bias"] is None else d["attention_bias"].shape[1])
    total = inp["total_sequence_length"] if total is None else total
    nbytes = gqa.gqa_workspace_size(dims, total, inp["local_window_size"])
    ws = torch.empty(max(nbytes + workspace_pad, 256), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)  # the contents on entry must not matter
    st = gqa.gqa_forward(dims, d["query"], d["key"], d["value"], d["k_buf"], d["v_buf"], d["k_buf"], d["v_buf"],
                         d["seqlens_k"], total, d["cos"], d["sin"], inp["scale"], inp["local_window_size"],
                         d["attention_bias"], out, ws, ws.numel(), stream)
    dst = gqa.gqa_check_device_status(stream)
    return st, dst, out.cpu(), d["k_buf"].cpu(), d["v_buf"].cpu()


def run_oracle(inp: dict, batches=None, heads=None, **kw):
    w = inp["workload"]
    a = dict(query=W.bits(inp["query"]), key=W.bits(inp["key"]), value=W.bits(inp["value"]),
             k_buf=W.bits(inp["k_buf"]), v_buf=W.bits(inp["v_buf"]), seqlens_k=inp["seqlens_k"].numpy(),
             total_sequence_length=inp["total_sequence_length"],
             cos_cache=None if inp["cos"] is None else W.bits(inp["cos"]),
             sin_cache=None if inp["sin"] is None else W.bits(inp["sin"]),
             num_heads=w.num_heads, kv_num_heads=w.kv_num_heads, scale=inp["scale"],
             local_window_size=inp["local_window_size"],
             attention_bias=None if inp["attention_bias"] is None else W.bits(inp["attention_bias"]),
             dtype=w.dtype, batches=batches, heads=heads)
    if inp.get("rotary_interleaved", 0):
        a["interleaved"] = True
    a.update(kw)
    return oracle.gqa_forward(**a)


def compare(inp: dict, cuda_res, oracle_res, heads=None, batches=None):
    """Asserts bit-exact buffers and the output within the dtype's tolerance.
    Returns the max abs error over the compared output elements."""
    w = inp["workload"]
    st, dst, out, kb, vb = cuda_res
    ost, oout, okb, ovb = oracle_res
    assert st == gqa.GQA_OK, gqa.gqa_status_string(st)
    assert dst == gqa.GQA_OK, gqa.gqa_status_string(dst)
    assert ost == oracle.STATUS_OK
    assert np.array_equal(W.bits(kb), okb), "key buffer differs from the oracle"
    assert np.array_equal(W.bits(vb), ovb), "value buffer differs from the oracle"
    B, S, H, D = w.batch, w.seq_len, w.num_heads, w.head_size
    got = out.float().numpy().astype(np.float64).reshape(B, S, H, D)
    ref = oout.reshape(B, S, H, D)
    bs = list(range(B)) if batches is None else list(batches)
    hs = list(range(H)) if heads is None else list(heads)
    g = got[bs][:, :, hs]
    r = ref[bs][:, :, hs]
    assert np.all(np.isfinite(g)), "non-finite output"
    e = np.abs(g - r)
    bound = np.maximum(TOL[w.dtype], ulp(r, w.dtype))
    worst = np.unravel_index(np.argmax(e - bound), e.shape)
    assert np.all(e <= bound), (f"error {e[worst]:.4e} > bound {bound[worst]:.4e} at {worst}: "
                                f"gpu {g[worst]:.6f} oracle {r[worst]:.6f}")
    return float(e.max())


def ulp(x, dtype):
    """One unit in the last place of T at |x| (normal range)."""
    bits = 10 if dtype == "fp16" else 7
    ax = np.maximum(np.abs(x), np.finfo(np.float64).tiny)
    return np.exp2(np.floor(np.log2(ax)) - bits)
