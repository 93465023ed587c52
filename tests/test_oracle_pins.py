"""Pins for the CPU oracle: each test checks it against something other than
itself -- hand-derived values, closed forms, invariants, a library routine
that computes a special case, or brute force on tiny inputs."""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from shared_kv_cache_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _tbits(x, dtype):
    """float array -> T bits via torch's own conversion (an independent routine)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(W.DTYPES[dtype])
    return W.bits(t)


# ---------------------------------------------------------------------------
# Rounding
# ---------------------------------------------------------------------------
def test_rounding_golden():
    n = 0
    for line in open(os.path.join(GOLDEN, "ieee_rounding.txt")):
        if line.startswith("#") or not line.strip():
            continue
        dt, f32hex, thex = line.split()[:3]
        x = np.array([int(f32hex, 16)], dtype=np.uint32).view(np.float32)
        got = int(oracle.f32_to_t(x, dt)[0])
        assert got == int(thex, 16), (line, hex(got))
        n += 1
    assert n >= 16


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_rounding_matches_torch(dtype):
    r = _rng(1)
    x = np.concatenate([r.standard_normal(200000).astype(np.float32) * s for s in (1e-6, 1.0, 3e3)])
    # values straddling exact halves
    mid = oracle.t_to_f32(r.integers(0, 0x7B00, 5000).astype(np.uint16), dtype)
    x = np.concatenate([x, mid, np.nextafter(mid, np.float32(np.inf)), np.nextafter(mid, np.float32(-np.inf))])
    assert np.array_equal(oracle.f32_to_t(x, dtype), _tbits(x, dtype))
    # widening is exact and inverts the narrowing on representable values
    b = r.integers(0, 0x7B00, 10000).astype(np.uint16)
    assert np.array_equal(oracle.f32_to_t(oracle.t_to_f32(b, dtype), dtype), b)


# ---------------------------------------------------------------------------
# Rotary embedding
# ---------------------------------------------------------------------------
def test_rotary_golden_closed_form():
    fix = {"fp16": ("3853", "3ABB"), "bf16": ("3F0A", "3F57")}
    for line in open(os.path.join(GOLDEN, "rotary_closed_form.txt")):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        dt, p, idx = f[0], int(f[1]), int(f[2])
        want = [int(h, 16) for h in f[3:11]]
        one = int(oracle.f32_to_t(np.float32(1.0), dt))
        cos = np.full((2, 4), one, np.uint16)
        sin = np.zeros((2, 4), np.uint16)
        cos[1, 0] = int(fix[dt][0], 16)
        sin[1, 0] = int(fix[dt][1], 16)
        x = np.zeros((1, 1, 1, 8), np.uint16)
        x[0, 0, 0, idx] = one
        got = oracle.rotary(x, np.array([[p]]), cos, sin, dt)[0, 0, 0]
        assert [int(g) for g in got] == want, line


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_rotary_is_complex_rotation(dtype):
    """Pair (x[j], x[j+D/2]) as z = x[j] + i x[j+D/2]; the rotary output is
    z * (cos + i sin), rounded to T (within one unit in the last place)."""
    r = _rng(2)
    B, S, Hh, D, rows = 2, 5, 3, 16, 40
    x = _tbits(r.standard_normal((B, S, Hh, D)), dtype)
    cos, sin = W.rotary_cache(rows, D, dtype)
    cos, sin = W.bits(cos), W.bits(sin)
    past = np.array([3, 17])
    pos = oracle.positions(past, S)
    y = oracle.t_to_f64(oracle.rotary(x, pos, cos, sin, dtype), dtype)
    xf = oracle.t_to_f64(x, dtype)
    c = oracle.t_to_f64(cos, dtype)[pos][:, :, None, :]
    s = oracle.t_to_f64(sin, dtype)[pos][:, :, None, :]
    z = (xf[..., : D // 2] + 1j * xf[..., D // 2:]) * (c + 1j * s)
    exact = np.concatenate([z.real, z.imag], axis=-1)
    ulp = np.spacing(np.abs(exact).astype(np.float16 if dtype == "fp16" else np.float32)).astype(np.float64)
    if dtype == "bf16":
        ulp = ulp * 2 ** 16
    assert np.all(np.abs(y - exact) <= ulp + 1e-30)
    # positions: token i of sequence b uses cache row past_b + i
    assert pos.tolist() == [[3, 4, 5, 6, 7], [17, 18, 19, 20, 21]]


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_rotary_interleaved_is_complex_rotation(dtype):
    """Interleaved layout: pair j is z = x[2j] + i x[2j+1], rotated by
    cos + i sin of cache entry j."""
    r = _rng(4)
    B, S, Hh, D = 1, 3, 2, 16
    x = _tbits(r.standard_normal((B, S, Hh, D)), dtype)
    cos, sin = W.rotary_cache(32, D, dtype)
    cos, sin = W.bits(cos), W.bits(sin)
    pos = oracle.positions(np.array([7]), S)
    y = oracle.t_to_f64(oracle.rotary(x, pos, cos, sin, dtype, interleaved=True), dtype)
    xf = oracle.t_to_f64(x, dtype)
    c = oracle.t_to_f64(cos, dtype)[pos][:, :, None, :]
    s = oracle.t_to_f64(sin, dtype)[pos][:, :, None, :]
    z = (xf[..., 0::2] + 1j * xf[..., 1::2]) * (c + 1j * s)
    exact = np.empty_like(xf)
    exact[..., 0::2] = z.real
    exact[..., 1::2] = z.imag
    ulp = np.spacing(np.abs(exact).astype(np.float16 if dtype == "fp16" else np.float32)).astype(np.float64)
    if dtype == "bf16":
        ulp = ulp * 2 ** 16
    assert np.all(np.abs(y - exact) <= ulp + 1e-30)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_rotary_position_zero_identity_and_norm(dtype):
    r = _rng(3)
    D = 128
    x = _tbits(r.standard_normal((1, 4, 2, D)), dtype)
    cos, sin = W.rotary_cache(64, D, dtype)
    cos, sin = W.bits(cos), W.bits(sin)
    y0 = oracle.rotary(x, np.zeros((1, 4), np.int64), cos, sin, dtype)
    assert np.array_equal(y0, x)
    pos = np.array([[1, 9, 33, 63]])
    y = oracle.t_to_f64(oracle.rotary(x, pos, cos, sin, dtype), dtype)
    xf = oracle.t_to_f64(x, dtype)
    # |c + i s| = 1 only up to the cache's rounding; the pair norm is kept
    # within that rounding plus the output's
    eps = 2 ** -10 if dtype == "fp16" else 2 ** -7
    n0 = np.hypot(xf[..., :64], xf[..., 64:])
    n1 = np.hypot(y[..., :64], y[..., 64:])
    assert np.all(np.abs(n1 - n0) <= 2 * eps * n0 + 1e-6)


# ---------------------------------------------------------------------------
# Scatter-append
# ---------------------------------------------------------------------------
def _small_case(dtype="fp16", B=3, S=4, H=4, Hkv=2, D=8, M=24, past=(0, 5, 13), seed=5,
                bias=None, window=0, total=None, sentinel=True):
    w = W.Workload("t", dtype, B, S, H, Hkv, D, M, 0, 0, bias_shape=bias, local_window_size=window,
                   total_sequence_length=total, seed=seed)
    inp = W.make_inputs(w, sentinel=sentinel)
    inp["seqlens_k"] = __import__("torch").tensor(past, dtype=__import__("torch").int32)
    # refill the past region for the chosen lengths
    gen = torch.Generator().manual_seed(seed + 1)
    for name in ("k_buf", "v_buf"):
        buf = inp[name]
        if sentinel:
            buf.view(torch.int16).fill_(W.SENTINEL_BITS[dtype])
        else:
            buf.zero_()
        for b, n in enumerate(past):
            if n:
                buf[b, :, :n] = torch.randn(Hkv, n, D, generator=gen).to(W.DTYPES[dtype])
    t = total if total is not None else max(past) + S
    inp["total_sequence_length"] = t
    inp["cos"], inp["sin"] = W.rotary_cache(max(t, M), D, dtype)
    if bias is not None:
        inp["attention_bias"] = (torch.randn(bias[0], bias[1], S, t, generator=gen) * 0.5).to(W.DTYPES[dtype])
    return w, inp


def _run_oracle(w, inp, **kw):
    a = dict(query=W.bits(inp["query"]), key=W.bits(inp["key"]), value=W.bits(inp["value"]),
             k_buf=W.bits(inp["k_buf"]), v_buf=W.bits(inp["v_buf"]),
             seqlens_k=inp["seqlens_k"].numpy(), total_sequence_length=inp["total_sequence_length"],
             cos_cache=None if inp["cos"] is None else W.bits(inp["cos"]),
             sin_cache=None if inp["sin"] is None else W.bits(inp["sin"]),
             num_heads=w.num_heads, kv_num_heads=w.kv_num_heads, scale=inp["scale"],
             local_window_size=inp["local_window_size"],
             attention_bias=None if inp["attention_bias"] is None else W.bits(inp["attention_bias"]),
             dtype=w.dtype)
    a.update(kw)
    return oracle.gqa_forward(**a)


def test_append_equals_cat_construction():
    """For a contiguous past, the shared-buffer scatter equals the cat-based
    construction cat(past, new) of the earlier lowering."""
    w, inp = _small_case()
    st, _, kb, vb = _run_oracle(w, inp)
    assert st == oracle.STATUS_OK
    B, S, Hkv, D = w.batch, w.seq_len, w.kv_num_heads, w.head_size
    pos = oracle.positions(inp["seqlens_k"].numpy(), S)
    krot = oracle.rotary(W.bits(inp["key"]).reshape(B, S, Hkv, D), pos, W.bits(inp["cos"]),
                         W.bits(inp["sin"]), w.dtype)
    for b, pb in enumerate(inp["seqlens_k"].tolist()):
        past_k = W.bits(inp["k_buf"])[b, :, :pb]
        cat_k = np.concatenate([past_k, krot[b].transpose(1, 0, 2)], axis=1)
        assert np.array_equal(kb[b, :, :pb + S], cat_k)
        past_v = W.bits(inp["v_buf"])[b, :, :pb]
        cat_v = np.concatenate([past_v, W.bits(inp["value"]).reshape(B, S, Hkv, D)[b].transpose(1, 0, 2)], axis=1)
        assert np.array_equal(vb[b, :, :pb + S], cat_v)


def test_append_equals_torch_pad_scatter_and_leaves_other_slots():
    """The pad+scatter formulation (pad with zeros, scatter along the
    sequence axis at seqlens_k + i) through torch.scatter, and untouched
    sentinel slots beyond the new tokens."""
    w, inp = _small_case(sentinel=True)
    st, _, _, vb = _run_oracle(w, inp)
    B, S, Hkv, D, M = w.batch, w.seq_len, w.kv_num_heads, w.head_size, w.max_seq_len
    past = inp["seqlens_k"].to(torch.int64)
    total = inp["total_sequence_length"]
    vbuf = inp["v_buf"].view(torch.int16)
    padded = torch.zeros(B, Hkv, total, D, dtype=torch.int16)
    for b in range(B):
        padded[b, :, : int(past[b])] = vbuf[b, :, : int(past[b])]
    idx = (past[:, None] + torch.arange(S)[None, :])[:, None, :, None].expand(B, Hkv, S, D)
    new = inp["value"].view(torch.int16).reshape(B, S, Hkv, D).permute(0, 2, 1, 3)
    scattered = padded.scatter(2, idx, new)
    for b in range(B):
        L = int(past[b]) + S
        assert np.array_equal(vb[b, :, :L].view(np.int16), scattered[b, :, :L].numpy())
        assert np.all(vb[b, :, L:] == W.SENTINEL_BITS[w.dtype])
    # every slot outside [past_b, past_b + S) keeps its bits
    before = W.bits(inp["v_buf"])
    for b in range(B):
        pb = int(past[b])
        assert np.array_equal(vb[b, :, :pb], before[b, :, :pb])
        assert np.array_equal(vb[b, :, pb + S:], before[b, :, pb + S:])


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------
def _sdpa_reference(w, inp, kb, vb):
    """Attention through torch's scaled_dot_product_attention in float64 with
    an explicit additive mask built as the pad+scatter lowering describes
    (k_pos <= past + q_pos -> 0, else -inf, shape [B, 1, S, kv_seq]) plus the
    bias, and the library's own grouped-query head mapping."""
    B, S, H, Hkv, D = w.batch, w.seq_len, w.num_heads, w.kv_num_heads, w.head_size
    past = inp["seqlens_k"].to(torch.int64)
    q = oracle.t_to_f64(W.bits(inp["query"]), w.dtype).reshape(B, S, H, D)
    pos = oracle.positions(past.numpy(), S)
    if inp["cos"] is not None:
        q = oracle.t_to_f64(oracle.rotary(W.bits(inp["query"]).reshape(B, S, H, D), pos,
                                          W.bits(inp["cos"]), W.bits(inp["sin"]), w.dtype), w.dtype)
    outs = []
    for b in range(B):
        L = int(past[b]) + S
        qb = torch.from_numpy(q[b]).permute(1, 0, 2)[None]           # [1, H, S, D]
        kk = torch.from_numpy(oracle.t_to_f64(kb[b, :, :L], w.dtype))[None]
        vv = torch.from_numpy(oracle.t_to_f64(vb[b, :, :L], w.dtype))[None]
        kpos = torch.arange(L)[None, :]
        qpos = (int(past[b]) + torch.arange(S))[:, None]
        keep = kpos <= qpos
        if inp["local_window_size"] > 0:
            keep &= kpos > qpos - inp["local_window_size"]
        mask = torch.zeros(S, L, dtype=torch.float64).masked_fill(~keep, float("-inf"))[None, None]
        if inp["attention_bias"] is not None:
            bias = torch.from_numpy(oracle.t_to_f64(W.bits(inp["attention_bias"]), w.dtype))
            bb = bias[b if bias.shape[0] > 1 else 0][None, :, :, :L]
            mask = mask + bb
        o = F.scaled_dot_product_attention(qb, kk, vv, attn_mask=mask, scale=float(np.float32(inp["scale"])),
                                           enable_gqa=(H != Hkv))
        outs.append(o[0].permute(1, 0, 2).reshape(S, H * D).numpy())
    return np.stack(outs)


@pytest.mark.parametrize("case", [
    dict(),
    dict(dtype="bf16", past=(7, 0, 11), seed=11),
    dict(bias=(1, 1), seed=12),
    dict(bias=(3, 4), seed=13),
    dict(window=3, seed=14),
    dict(window=5, bias=(1, 4), past=(9, 2, 20), seed=15),
    dict(H=6, Hkv=3, D=16, seed=16),
    dict(H=4, Hkv=4, seed=17),
    dict(S=1, past=(0, 9, 22), seed=18),
])
def test_attention_matches_sdpa(case):
    w, inp = _small_case(**case)
    st, out, kb, vb = _run_oracle(w, inp)
    assert st == oracle.STATUS_OK
    ref = _sdpa_reference(w, inp, kb, vb)
    assert np.abs(out - ref).max() < 1e-12


def test_attention_pure_python_brute_force():
    """Loops over every (b, h, i, j) with math.exp, on a tiny case."""
    w, inp = _small_case(B=2, S=3, H=4, Hkv=2, D=8, M=12, past=(2, 5), bias=(2, 1), window=4, seed=21)
    st, out, kb, vb = _run_oracle(w, inp)
    B, S, H, Hkv, D = 2, 3, 4, 2, 8
    G = H // Hkv
    pos = oracle.positions(inp["seqlens_k"].numpy(), S)
    qr = oracle.t_to_f64(oracle.rotary(W.bits(inp["query"]).reshape(B, S, H, D), pos,
                                       W.bits(inp["cos"]), W.bits(inp["sin"]), w.dtype), w.dtype)
    K = oracle.t_to_f64(kb, w.dtype)
    V = oracle.t_to_f64(vb, w.dtype)
    bias = oracle.t_to_f64(W.bits(inp["attention_bias"]), w.dtype)
    scale = float(np.float32(inp["scale"]))
    for b in range(B):
        pb = int(inp["seqlens_k"][b])
        for h in range(H):
            for i in range(S):
                p = pb + i
                keys = [j for j in range(p + 1) if j > p - 4]
                z = []
                for j in keys:
                    d = sum(qr[b, i, h, t] * K[b, h // G, j, t] for t in range(D))
                    z.append(d * scale + bias[b, 0, i, j])
                mx = max(z)
                e = [math.exp(x - mx) for x in z]
                tot = sum(e)
                for t in range(D):
                    o = sum(e[n] / tot * V[b, h // G, j, t] for n, j in enumerate(keys))
                    assert abs(o - out[b, i, h * D + t]) < 1e-12


def test_uniform_attention_closed_form():
    """With q = 0 (and no rotary) every visible key has the same score, so
    each output row is the mean of the visible value rows; this fixes the
    causal bound and the window bound exactly."""
    for window in (0, 1, 3):
        w, inp = _small_case(window=window, seed=30 + window)
        inp["query"].zero_()
        inp["cos"] = inp["sin"] = None
        st, out, kb, vb = _run_oracle(w, inp)
        V = oracle.t_to_f64(vb, w.dtype)
        B, S, H, Hkv, D = w.batch, w.seq_len, w.num_heads, w.kv_num_heads, w.head_size
        for b in range(B):
            pb = int(inp["seqlens_k"][b])
            for i in range(S):
                p = pb + i
                lo = 0 if window <= 0 else max(0, p - window + 1)
                for h in range(H):
                    mean = V[b, h // (H // Hkv), lo:p + 1].mean(axis=0)
                    assert np.abs(out[b, i, h * D:(h + 1) * D] - mean).max() < 1e-12


def test_window_one_returns_current_value_and_large_window_is_full():
    w, inp = _small_case(window=1, seed=40)
    st, out, kb, vb = _run_oracle(w, inp)
    B, S, H, Hkv, D = w.batch, w.seq_len, w.num_heads, w.kv_num_heads, w.head_size
    vnew = oracle.t_to_f64(W.bits(inp["value"]), w.dtype).reshape(B, S, Hkv, D)
    for h in range(H):
        assert np.array_equal(out[:, :, h * D:(h + 1) * D], vnew[:, :, h // (H // Hkv)])
    w2, inp2 = _small_case(window=0, seed=40)
    w3, inp3 = _small_case(window=10 ** 6, seed=40)
    assert np.array_equal(_run_oracle(w2, inp2)[1], _run_oracle(w3, inp3)[1])


def test_bias_indexing_closed_form():
    """q = 0 and a bias of +60 at one absolute key position j* for query row
    i (and 0 elsewhere): the output row is v[j*] up to e^-60."""
    w, inp = _small_case(bias=(3, 4), seed=50, past=(4, 6, 9))
    inp["query"].zero_()
    inp["cos"] = inp["sin"] = None
    bias = torch.zeros_like(inp["attention_bias"], dtype=torch.float32)
    picks = {}
    for b in range(3):
        for h in range(4):
            for i in range(w.seq_len):
                j = (b * 7 + h * 3 + i * 5) % (int(inp["seqlens_k"][b]) + i + 1)
                bias[b, h, i, j] = 60.0
                picks[(b, h, i)] = j
    inp["attention_bias"] = bias.to(W.DTYPES[w.dtype])
    st, out, kb, vb = _run_oracle(w, inp)
    V = oracle.t_to_f64(vb, w.dtype)
    D = w.head_size
    for (b, h, i), j in picks.items():
        assert np.abs(out[b, i, h * D:(h + 1) * D] - V[b, h // 2, j]).max() < 1e-20


def test_probability_rows_sum_to_one():
    w, inp = _small_case(bias=(1, 1), window=6, seed=60)
    B, S, H, D = w.batch, w.seq_len, w.num_heads, w.head_size
    _, _, kb, vb = _run_oracle(w, inp)
    q = W.bits(inp["query"]).reshape(B, S, H, D)
    _, probs = oracle.attention(q, kb, vb, inp["seqlens_k"].numpy(), H, w.kv_num_heads,
                                inp["scale"], 6, W.bits(inp["attention_bias"]), w.dtype,
                                return_probs=True)
    for P in probs.values():
        assert np.all(np.abs(P.sum(axis=1) - 1.0) < 1e-14)
        assert np.all(P >= 0)


def test_default_scale_is_inverse_sqrt_head_size():
    w, inp = _small_case(seed=70, D=16)
    a = _run_oracle(w, inp, scale=0.0)[1]
    b = _run_oracle(w, inp, scale=1.0 / math.sqrt(16))[1]
    assert np.array_equal(a, b)


def test_decode_equals_last_row_of_prefill():
    """Prefill S+1 tokens at once versus prefill S then decode 1: the decode
    output equals the last prefill row, and the buffers are bit-equal."""
    for dtype in ("fp16", "bf16"):
        w, inp = _small_case(dtype=dtype, S=5, past=(0, 3, 8), seed=80)
        B, S, Hkv, D, H = w.batch, 5, w.kv_num_heads, w.head_size, w.num_heads
        st, full, kb_full, vb_full = _run_oracle(w, inp)
        first = dict(inp)
        for n in ("query", "key", "value"):
            first[n] = inp[n][:, :4].contiguous()
        w4 = w.with_(seq_len=4)
        st1, out4, kb1, vb1 = _run_oracle(w4, first)
        second = dict(inp)
        for n in ("query", "key", "value"):
            second[n] = inp[n][:, 4:].contiguous()
        second["k_buf"] = torch.from_numpy(kb1.view(np.int16)).view(W.DTYPES[dtype])
        second["v_buf"] = torch.from_numpy(vb1.view(np.int16)).view(W.DTYPES[dtype])
        second["seqlens_k"] = inp["seqlens_k"] + 4
        st2, out1, kb2, vb2 = _run_oracle(w.with_(seq_len=1), second)
        assert st1 == st2 == oracle.STATUS_OK
        assert np.array_equal(kb2, kb_full) and np.array_equal(vb2, vb_full)
        assert np.abs(out1[:, 0] - full[:, 4]).max() < 1e-12
        assert np.abs(out4 - full[:, :4]).max() < 1e-12


def test_kv_cache_example_shapes():
    """The worked shapes of the rocMLIR "KV Cache" example (prefill 32 x 8,
    then one decode token over 33 keys in a buffer of max_seq_len)."""
    for line in open(os.path.join(GOLDEN, "kv_cache_example_shapes.txt")):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        S, past, D, M, sr, sc, orow, ocol = map(int, f[1:])
        w = W.Workload("ex", "fp16", 1, S, 1, 1, D, M, past, past, seed=90)
        inp = W.make_inputs(w)
        B = 1
        _, _, kb, vb = _run_oracle(w, inp)
        q = oracle.rotary(W.bits(inp["query"]).reshape(1, S, 1, D), oracle.positions(np.array([past]), S),
                          W.bits(inp["cos"]), W.bits(inp["sin"]), "fp16")
        out, probs = oracle.attention(q, kb, vb, np.array([past]), 1, 1, inp["scale"], 0, None, "fp16",
                                      return_probs=True)
        assert probs[(0, 0)].shape == (sr, sc)
        assert out[0, :, 0, :].shape == (orow, ocol)


def test_mha_special_case_and_head_mapping():
    """kv_num_heads == num_heads is plain multi-head attention; with G > 1,
    query head h equals a single-head run against KV head h // G."""
    w, inp = _small_case(H=4, Hkv=4, seed=100)
    st, out, kb, vb = _run_oracle(w, inp)
    assert np.abs(out - _sdpa_reference(w, inp, kb, vb)).max() < 1e-12
    w, inp = _small_case(H=6, Hkv=2, D=8, seed=101)
    st, out, kb, vb = _run_oracle(w, inp)
    B, S, D = w.batch, w.seq_len, w.head_size
    q = oracle.rotary(W.bits(inp["query"]).reshape(B, S, 6, D), oracle.positions(inp["seqlens_k"].numpy(), S),
                      W.bits(inp["cos"]), W.bits(inp["sin"]), w.dtype)
    for h in range(6):
        one = oracle.attention(q[:, :, h:h + 1], kb[:, h // 3:h // 3 + 1], vb[:, h // 3:h // 3 + 1],
                               inp["seqlens_k"].numpy(), 1, 1, float(np.float32(inp["scale"])), 0, None, w.dtype)
        assert np.array_equal(one[:, :, 0], out[:, :, h * D:(h + 1) * D])


# ---------------------------------------------------------------------------
# Overflow
# ---------------------------------------------------------------------------
def test_overflow_returns_error_and_leaves_buffers():
    w, inp = _small_case(M=24, past=(0, 5, 21), total=24, seed=110)   # 21 + 4 > 24
    st, out, kb, vb = _run_oracle(w, inp)
    assert st == oracle.STATUS_KV_OVERFLOW and out is None
    assert np.array_equal(kb, W.bits(inp["k_buf"])) and np.array_equal(vb, W.bits(inp["v_buf"]))
    # total_sequence_length beyond the buffer
    w, inp = _small_case(M=24, past=(0, 5, 13), seed=111)
    st, *_ = _run_oracle(w, inp, total_sequence_length=25)
    assert st == oracle.STATUS_KV_OVERFLOW
    # exactly full is fine
    w, inp = _small_case(M=24, past=(0, 5, 20), seed=112)
    assert _run_oracle(w, inp)[0] == oracle.STATUS_OK
    # a length beyond total_sequence_length but inside the buffer is invalid
    w, inp = _small_case(M=24, past=(0, 5, 13), seed=113)
    assert _run_oracle(w, inp, total_sequence_length=16)[0] == oracle.STATUS_INVALID_ARGUMENT


# ---------------------------------------------------------------------------
# Non-shared binding: separate past and present buffers, present = past + new
# ---------------------------------------------------------------------------
def _split_binding(w, inp, Mp, seed):
    """The case's past rows moved into separate past buffers of Mp slots
    (slots from past_b on hold other random rows, not part of the past) and
    present buffers that start as the sentinel."""
    B, Hkv, D = w.batch, w.kv_num_heads, w.head_size
    gen = torch.Generator().manual_seed(seed)
    past, present = {}, {}
    for name in ("k_buf", "v_buf"):
        pk = torch.randn(B, Hkv, Mp, D, generator=gen).to(W.DTYPES[w.dtype])
        for b, n in enumerate(inp["seqlens_k"].tolist()):
            pk[b, :, :min(n, Mp)] = inp[name][b, :, :min(n, Mp)]
        past[name] = W.bits(pk)
        present[name] = np.full(W.bits(inp[name]).shape, W.SENTINEL_BITS[w.dtype], dtype=np.uint16)
    return past, present


def _run_split(w, inp, past, present):
    return _run_oracle(w, inp, k_buf=present["k_buf"], v_buf=present["v_buf"], past_key=past["k_buf"],
                       past_value=past["v_buf"])


def test_non_shared_present_is_past_then_new():
    """Per sequence the present holds cat(past[:past_b], new rows) -- built
    here with torch.cat from the raw value rows -- and every later slot keeps
    its bits; the output is exactly the shared binding's on a buffer that
    holds the same past."""
    w, inp = _small_case(sentinel=True, seed=120)
    B, S, Hkv, D = w.batch, w.seq_len, w.kv_num_heads, w.head_size
    past, present = _split_binding(w, inp, Mp=max(inp["seqlens_k"].tolist()) + 3, seed=121)
    st, out, kb, vb = _run_split(w, inp, past, present)
    st2, out2, kb2, _ = _run_oracle(w, inp)
    assert st == st2 == oracle.STATUS_OK
    assert np.array_equal(out, out2)
    new_v = inp["value"].view(torch.int16).reshape(B, S, Hkv, D)
    for b, pb in enumerate(inp["seqlens_k"].tolist()):
        L = pb + S
        cat_v = torch.cat([torch.from_numpy(past["v_buf"][b, :, :pb].view(np.int16)), new_v[b].transpose(0, 1)], dim=1)
        assert np.array_equal(vb[b, :, :L].view(np.int16), cat_v.numpy())
        assert np.array_equal(kb[b, :, :L], kb2[b, :, :L])  # rotated keys as in the shared binding
        assert np.all(kb[b, :, L:] == W.SENTINEL_BITS[w.dtype]) and np.all(vb[b, :, L:] == W.SENTINEL_BITS[w.dtype])


def test_non_shared_ignores_past_beyond_its_length():
    """Past slots from past_b on are not part of the past: changing them
    changes neither the output nor the present."""
    w, inp = _small_case(sentinel=True, seed=122)
    Mp = max(inp["seqlens_k"].tolist()) + 5
    past, present = _split_binding(w, inp, Mp, seed=123)
    st, out, kb, vb = _run_split(w, inp, past, present)
    for name in ("k_buf", "v_buf"):
        for b, pb in enumerate(inp["seqlens_k"].tolist()):
            past[name][b, :, pb:] ^= 0x1234
    st2, out2, kb2, vb2 = _run_split(w, inp, past, present)
    assert st == st2 == oracle.STATUS_OK
    assert np.array_equal(out, out2) and np.array_equal(kb, kb2) and np.array_equal(vb, vb2)


def test_non_shared_past_shorter_than_a_length_is_invalid():
    w, inp = _small_case(sentinel=True, seed=124, past=(0, 5, 13))
    past, present = _split_binding(w, inp, Mp=13, seed=125)
    assert _run_split(w, inp, past, present)[0] == oracle.STATUS_OK     # past_b == Mp is fine
    past, present = _split_binding(w, inp, Mp=12, seed=125)
    st, out, kb, vb = _run_split(w, inp, past, present)
    assert st == oracle.STATUS_INVALID_ARGUMENT and out is None
    assert np.array_equal(kb, present["k_buf"]) and np.array_equal(vb, present["v_buf"])
