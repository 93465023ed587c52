"""Pins for the oracle's operator variants: packed QKV input and the
sliding-window cache with contiguous eviction.

Packed QKV follows the [batch, seq, hidden] -> [batch, seq, heads, head_size]
reading of the torch-mlir PR description ("[TorchOnnxToTorch] Add
pad+scatter KV cache and mask to GQA"); the eviction follows the SWA
follow-up of "Clarification about GroupQueryAttention behavior" (keep only
the min(total_sequence_length, cache_capacity) most recent tokens,
contiguously).  Each test checks the oracle against something other than
itself: torch's concatenation, position-coded rows, brute force with
math.exp, and attention over the unbounded history."""
import math

import numpy as np
import pytest
import torch

import oracle
from shared_kv_cache_gb300 import workloads as W


def _bits(t):
    return W.bits(t)


def _rand(shape, gen, dtype):
    return torch.randn(*shape, generator=gen).to(W.DTYPES[dtype])


# ---------------------------------------------------------------------------
# Packed QKV
# ---------------------------------------------------------------------------
def test_unpack_follows_token_major_head_layout():
    """Packing built with torch.cat over the head axis of [B, S, heads, D]
    views comes apart into exactly the three inputs."""
    gen = torch.Generator().manual_seed(1)
    B, S, H, Hkv, D = 2, 3, 6, 2, 8
    q, k, v = (_rand((B, S, n * D), gen, "fp16") for n in (H, Hkv, Hkv))
    packed = torch.cat([q.view(B, S, H, D), k.view(B, S, Hkv, D), v.view(B, S, Hkv, D)], dim=2).reshape(B, S, -1)
    uq, uk, uv = oracle.unpack_qkv(_bits(packed), H, Hkv)
    assert np.array_equal(uq, _bits(q)) and np.array_equal(uk, _bits(k)) and np.array_equal(uv, _bits(v))
    # token 1, value head 1, element 5 sits at (H + Hkv + 1) * D + 5 of row (0, 1)
    assert _bits(packed)[0, 1, (H + Hkv + 1) * D + 5] == _bits(v)[0, 1, D + 5]


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_packed_call_equals_separate_inputs(dtype):
    gen = torch.Generator().manual_seed(2)
    B, S, H, Hkv, D, M = 2, 4, 4, 2, 8, 16
    past = np.array([3, 9])
    q, k, v = (_rand((B, S, n * D), gen, dtype) for n in (H, Hkv, Hkv))
    kb, vb = (_bits(_rand((B, Hkv, M, D), gen, dtype)) for _ in range(2))
    cos, sin = W.rotary_cache(M, D, dtype)
    common = dict(k_buf=kb, v_buf=vb, seqlens_k=past, total_sequence_length=13, cos_cache=_bits(cos),
                  sin_cache=_bits(sin), num_heads=H, kv_num_heads=Hkv, scale=0.0, local_window_size=0,
                  attention_bias=None, dtype=dtype)
    a = oracle.gqa_forward(_bits(q), _bits(k), _bits(v), **common)
    packed = torch.cat([q.view(B, S, H, D), k.view(B, S, Hkv, D), v.view(B, S, Hkv, D)], dim=2).reshape(B, S, -1)
    b = oracle.gqa_forward(_bits(packed), None, None, **common)
    assert a[0] == b[0] == oracle.STATUS_OK
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2]) and np.array_equal(a[3], b[3])


# ---------------------------------------------------------------------------
# Sliding-window cache with contiguous eviction
# ---------------------------------------------------------------------------
def _call(q, k, v, kb, vb, past, total, cos, sin, H, Hkv, window, dtype, evict, bias=None):
    return oracle.gqa_forward(q, k, v, kb, vb, np.asarray(past), total, cos, sin, H, Hkv, 0.0, window, bias, dtype,
                              evict=evict)


def test_evicting_mode_without_overflow_is_the_plain_append():
    gen = torch.Generator().manual_seed(3)
    B, S, H, Hkv, D, M = 3, 4, 4, 2, 8, 24
    past = [0, 5, 20]           # 20 + 4 = 24: exactly full, nothing evicted
    q, k, v = (_bits(_rand((B, S, n * D), gen, "fp16")) for n in (H, Hkv, Hkv))
    kb, vb = (_bits(_rand((B, Hkv, M, D), gen, "fp16")) for _ in range(2))
    cos, sin = (_bits(t) for t in W.rotary_cache(M, D, "fp16"))
    a = _call(q, k, v, kb, vb, past, 24, cos, sin, H, Hkv, 0, "fp16", False)
    b = _call(q, k, v, kb, vb, past, 24, cos, sin, H, Hkv, 0, "fp16", True)
    assert a[0] == b[0] == oracle.STATUS_OK
    assert np.array_equal(a[2], b[2]) and np.array_equal(a[3], b[3])
    assert np.abs(a[1] - b[1]).max() < 1e-12


def test_eviction_keeps_the_most_recent_tokens_contiguously():
    """Rows coded with their absolute position: after the call slot s holds
    position P + S - n_keep + s, n_keep = min(P + S, M); later slots keep
    their bits."""
    B, S, Hkv, D, M = 4, 3, 2, 8, 8
    past = [2, 5, 7, 30]        # n_old = 2, 5, 7, 8; P + S = 5, 8, 10, 33
    sentinel = W.SENTINEL_BITS["fp16"]

    def row(pos):               # a row whose every element is the position (exact in fp16)
        return _bits(torch.full((D,), float(pos), dtype=torch.float16))

    buf = np.full((B, Hkv, M, D), sentinel, dtype=np.uint16)
    new = np.zeros((B, S, Hkv, D), dtype=np.uint16)
    for b, P in enumerate(past):
        n_old = min(P, M)
        for s in range(n_old):
            buf[b, :, s] = row(P - n_old + s)
        for i in range(S):
            new[b, i, :] = row(P + i)
    out = oracle.evict_keep_recent(buf, new, np.array(past))
    for b, P in enumerate(past):
        n_keep = min(P + S, M)
        for s in range(n_keep):
            assert np.all(out[b, :, s] == row(P + S - n_keep + s)), (b, s)
        assert np.all(out[b, :, n_keep:] == sentinel)


@pytest.mark.parametrize("S,window,dtype", [(1, 8, "fp16"), (1, 5, "bf16"), (3, 6, "fp16"), (2, 7, "bf16")])
def test_eviction_equals_windowed_attention_over_the_whole_history(S, window, dtype):
    """Generating T tokens S at a time into a cache of M = 8 slots with a
    window that fits it (W <= M - S + 1) gives, at every step, the output of
    the plain operator over an unbounded buffer holding the whole history,
    and the cache holds that buffer's last n_keep rows bit for bit (so the
    keys were rotated at their absolute positions)."""
    gen = torch.Generator().manual_seed(10 + S + window)
    B, H, Hkv, D, M, T = 2, 4, 2, 8, 8, 24
    sentinel = W.SENTINEL_BITS[dtype]
    cos, sin = (_bits(t) for t in W.rotary_cache(T, D, dtype))
    kc = np.full((B, Hkv, M, D), sentinel, dtype=np.uint16)
    vc = kc.copy()
    ku = np.full((B, Hkv, T, D), sentinel, dtype=np.uint16)
    vu = ku.copy()
    for t0 in range(0, T, S):
        q, k, v = (_bits(_rand((B, S, n * D), gen, dtype)) for n in (H, Hkv, Hkv))
        past = [t0, t0]
        st_c, out_c, kc, vc = _call(q, k, v, kc, vc, past, t0 + S, cos, sin, H, Hkv, window, dtype, True)
        st_u, out_u, ku, vu = _call(q, k, v, ku, vu, past, t0 + S, cos, sin, H, Hkv, window, dtype, False)
        assert st_c == st_u == oracle.STATUS_OK
        assert np.abs(out_c - out_u).max() < 1e-12
        n_keep = min(t0 + S, M)
        assert np.array_equal(kc[:, :, :n_keep], ku[:, :, t0 + S - n_keep:t0 + S])
        assert np.array_equal(vc[:, :, :n_keep], vu[:, :, t0 + S - n_keep:t0 + S])


def test_eviction_full_attention_brute_force():
    """No window: every query sees the cached tokens and the new ones up to
    itself, with the bias read at the absolute key position.  Pure-Python
    loops with math.exp."""
    gen = torch.Generator().manual_seed(20)
    B, S, H, Hkv, D, M, total = 2, 2, 2, 1, 4, 5, 11
    past = [3, 9]                  # n_old = 3 and 5
    q, k, v = (_bits(_rand((B, S, n * D), gen, "bf16")) for n in (H, Hkv, Hkv))
    kb, vb = (_bits(_rand((B, Hkv, M, D), gen, "bf16")) for _ in range(2))
    bias = _bits((torch.randn(1, 1, S, total, generator=gen) * 0.5).to(torch.bfloat16))
    cos, sin = (_bits(t) for t in W.rotary_cache(total, D, "bf16"))
    st, out, _, _ = _call(q, k, v, kb, vb, past, total, cos, sin, H, Hkv, 0, "bf16", True, bias=bias)
    assert st == oracle.STATUS_OK
    pos = oracle.positions(np.array(past), S)
    qr = oracle.t_to_f64(oracle.rotary(q.reshape(B, S, H, D), pos, cos, sin, "bf16"), "bf16")
    kr = oracle.t_to_f64(oracle.rotary(k.reshape(B, S, Hkv, D), pos, cos, sin, "bf16"), "bf16")
    vn = oracle.t_to_f64(v.reshape(B, S, Hkv, D), "bf16")
    K, V = oracle.t_to_f64(kb, "bf16"), oracle.t_to_f64(vb, "bf16")
    bf = oracle.t_to_f64(bias, "bf16")
    scale = float(np.float32(1.0 / math.sqrt(D)))
    for b, P in enumerate(past):
        n_old = min(P, M)
        first = P - n_old

        def key(j):
            return (K[b, 0, j - first], V[b, 0, j - first]) if j < P else (kr[b, j - P, 0], vn[b, j - P, 0])
        for i in range(S):
            p = P + i
            keys = list(range(first, p + 1))
            for h in range(H):
                z = [sum(qr[b, i, h, t] * key(j)[0][t] for t in range(D)) * scale + bf[0, 0, i, j] for j in keys]
                mx = max(z)
                e = [math.exp(x - mx) for x in z]
                tot = sum(e)
                for t in range(D):
                    o = sum(e[n] / tot * key(j)[1][t] for n, j in enumerate(keys))
                    assert abs(o - out[b, i, h * D + t]) < 1e-12


def test_eviction_statuses():
    """The evicting buffer always has room; a past length beyond
    total_sequence_length (or negative) stays an invalid argument, and
    without eviction the same call overflows."""
    S, M = 4, 8
    assert oracle.check_lengths([30], S, M, 34, evict=True) == oracle.STATUS_OK
    assert oracle.check_lengths([30], S, M, 34, evict=False) == oracle.STATUS_KV_OVERFLOW
    assert oracle.check_lengths([31], S, M, 34, evict=True) == oracle.STATUS_INVALID_ARGUMENT
    assert oracle.check_lengths([-1], S, M, 34, evict=True) == oracle.STATUS_INVALID_ARGUMENT
    with pytest.raises(ValueError):
        z = np.zeros((1, 1, 8), dtype=np.uint16)
        oracle.gqa_forward(z, z, z, np.zeros((1, 1, 8, 8), np.uint16), np.zeros((1, 1, 8, 8), np.uint16),
                           np.array([0]), 1, None, None, 1, 1, 0.0, 0, None, "fp16",
                           past_key=np.zeros((1, 1, 4, 8), np.uint16), past_value=np.zeros((1, 1, 4, 8), np.uint16),
                           evict=True)
