"""Host logic of the tensor-level API (no GPU): the per-shape plan cache and
the grow-only workspace."""
import torch

import shared_kv_cache_gb300 as gqa
from shared_kv_cache_gb300 import api


def _t(*shape, dtype=torch.float16):
    return torch.empty(*shape, dtype=dtype)


def test_plan_cache_per_shape_and_entry():
    gqa.load_library()
    ws = api.Workspace()
    q, k, kb = _t(2, 1, 8 * 64), _t(2, 1, 2 * 64), _t(2, 2, 128, 64)
    args = (q, k, kb, 8, 2, None, None, 0, 64, 0)
    dev = api._plan(ws, False, *args)
    assert api._plan(ws, False, *args) is dev            # cached
    host = api._plan(ws, True, *args)
    assert host is not dev and host[1] > dev[1]          # the host entry also stages the step's data
    assert dev[1] == gqa.gqa_workspace_size(dev[0], 64, 0)
    assert host[1] == gqa.gqa_workspace_size_host(host[0], 64, 0)
    # another shape, another plan; the cache is bounded
    for s in range(70):
        api._plan(ws, False, _t(2, 1 + s, 8 * 64), _t(2, 1 + s, 2 * 64), kb, 8, 2, None, None, 0, 64 + s, 0)
    assert len(ws.plans) <= 65


def test_workspace_grows_only():
    ws = api.Workspace()
    assert ws.get(0, "cpu") is None
    a = ws.get(1000, "cpu")
    assert a.numel() >= 1000
    assert ws.get(500, "cpu") is a                       # reused
    b = ws.get(5000, "cpu")
    assert b is not a and b.numel() >= 5000
