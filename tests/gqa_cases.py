"""Shared helpers for the tests: run one GroupQueryAttention call through the
C ABI on the GPU, and the same inputs through the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import shared_kv_cache_gb300 as gqa
from shared_kv_cache_gb300 import workloads as W

# Attention output tolerance: max-abs 2e-3 for fp16 and 1e-2 for bf16 against
# the oracle's float64 result.  A T output is at best the correctly rounded
# value, at most half a unit in the last place (ulp) from the exact one; where
# that half ulp alone exceeds the tolerance (bf16 |o| >= 4, fp16 |o| >= 8) no
# T output can meet it, and there the output must be faithfully rounded
# instead: less than one ulp of T from the exact value.
TOL = {"fp16": 2e-3, "bf16": 1e-2}


def to_device(inp: dict, device="cuda") -> dict:
    out = {}
    for k, v in inp.items():
        out[k] = v.to(device) if isinstance(v, torch.Tensor) else v
    return out


def pack_qkv(inp: dict) -> torch.Tensor:
    """The packed form of the case's new rows: per token its query heads,
    then its key heads, then its value heads ([B, S, (H + 2 Hkv) * D])."""
    w = inp["workload"]
    B, S, D = w.batch, w.seq_len, w.head_size
    parts = [inp["query"].view(B, S, w.num_heads, D), inp["key"].view(B, S, w.kv_num_heads, D),
             inp["value"].view(B, S, w.kv_num_heads, D)]
    return torch.cat(parts, dim=2).reshape(B, S, -1).contiguous()


def dims_of(inp: dict):
    w = inp["workload"]
    bias = inp["attention_bias"]
    return gqa.make_dims(w.batch, w.seq_len, w.num_heads, w.kv_num_heads, w.head_size, w.max_seq_len, w.dtype,
                         inp.get("rotary_interleaved", 0), 0 if inp["cos"] is None else inp["cos"].shape[0],
                         1 if bias is None else bias.shape[0], 1 if bias is None else bias.shape[1],
                         kv_eviction=inp.get("kv_eviction", 0))


def run_cuda(inp: dict, stream=None, total=None, workspace_pad=0, packed=False):
    """Returns (status, device_status, out[CPU], k_buf[CPU], v_buf[CPU]).
    packed: the new rows go in as one packed query tensor (key, value NULL)."""
    d = to_device(inp)
    out = torch.full_like(d["query"], float("nan"))
    dims = dims_of(inp)
    total = inp["total_sequence_length"] if total is None else total
    nbytes = gqa.gqa_workspace_size(dims, total, inp["local_window_size"])
    ws = torch.empty(max(nbytes + workspace_pad, 256), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)  # the contents on entry must not matter
    q, k, v = (pack_qkv(inp).cuda(), None, None) if packed else (d["query"], d["key"], d["value"])
    st = gqa.gqa_forward(dims, q, k, v, d["k_buf"], d["v_buf"], d["k_buf"], d["v_buf"],
                         d["seqlens_k"], total, d["cos"], d["sin"], inp["scale"], inp["local_window_size"],
                         d["attention_bias"], out, ws, ws.numel(), stream)
    dst = gqa.gqa_check_device_status(stream)
    return st, dst, out.cpu(), d["k_buf"].cpu(), d["v_buf"].cpu()


def custom(dtype="bf16", B=3, S=1, H=8, Hkv=2, D=128, M=1000, past=(0, 517, 999), seed=7, bias=None,
           window=0, total=None, rotary=True, interleaved=0, sentinel=True, evict=False):
    """A seeded case of any shape: per-sequence past lengths `past`, past rows
    N(0, 1), other slots the NaN sentinel; bias (Bb, Hb) ~ N(0, 0.5).  With
    `evict` the call uses the evicting sliding-window cache: a past length
    may exceed M, and the buffer holds that sequence's min(past, M) most
    recent rows."""
    w = W.Workload("custom", dtype, B, S, H, Hkv, D, M, 0, 0, bias_shape=bias, local_window_size=window,
                   total_sequence_length=total, rotary=rotary, seed=seed)
    inp = W.make_inputs(w, sentinel=sentinel, fill_past=False)
    inp["seqlens_k"] = torch.tensor(past, dtype=torch.int32)
    gen = torch.Generator().manual_seed(seed + 1000)
    for name in ("k_buf", "v_buf"):
        for b, n in enumerate(past):
            n = min(n, M)
            if n > 0:
                inp[name][b, :, :n] = torch.randn(Hkv, n, D, generator=gen).to(W.DTYPES[dtype])
    t = total if total is not None else max(past) + S
    inp["total_sequence_length"] = t
    if rotary:
        inp["cos"], inp["sin"] = W.rotary_cache(max(t, M), D, dtype)
    if bias is not None:
        inp["attention_bias"] = (torch.randn(bias[0], bias[1], S, t, generator=gen) * 0.5).to(W.DTYPES[dtype])
    inp["rotary_interleaved"] = interleaved
    inp["kv_eviction"] = 1 if evict else 0
    return inp


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
    if inp.get("kv_eviction", 0):
        a["evict"] = True
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
    ok, n_floor = within_tolerance(e, r, w.dtype)
    if not ok.all():
        u = ulp(r, w.dtype)
        excess = np.where(ok, -np.inf, e - np.where(0.5 * u > TOL[w.dtype], u, TOL[w.dtype]))
        worst = np.unravel_index(np.argmax(excess), e.shape)
        raise AssertionError(f"{int((~ok).sum())} outputs out of tolerance; worst error {e[worst]:.4e} at {worst}: "
                             f"gpu {g[worst]:.6f} oracle {r[worst]:.6f} (ulp {u[worst]:.3e})")
    if n_floor:
        print(f"[{w.name}] {n_floor} of {e.size} outputs above the range where {TOL[w.dtype]} is attainable "
              f"(checked for faithful rounding)")
    return float(e.max())


def within_tolerance(err, ref, dtype):
    """(ok mask, number of elements under the faithful-rounding rule).  Where
    half an ulp of T at the reference fits in the tolerance, the error must be
    within the tolerance; elsewhere it must be below one ulp."""
    u = ulp(ref, dtype)
    floor = 0.5 * u > TOL[dtype]
    ok = np.where(floor, err < u, err <= TOL[dtype])
    return ok, int(floor.sum())


def ulp(x, dtype):
    """One unit in the last place of T at |x| (normal range)."""
    bits = 10 if dtype == "fp16" else 7
    ax = np.maximum(np.abs(x), np.finfo(np.float64).tiny)
    _, e = np.frexp(ax)             # ax = m * 2^e, m in [0.5, 1): exact, unlike log2 near a power of two
    return np.ldexp(1.0, e - 1 - bits)
