"""NVTX ranges around the Python entry points (FA_NVTX): each call pushes one
named range and pops it again, also when the call raises."""
import pytest
import torch

import exact_attention_42_gb300 as fa
from exact_attention_42_gb300 import api


def test_ranges_are_balanced_and_named(monkeypatch):
    events = []
    monkeypatch.setattr(api, "NVTX", True)
    monkeypatch.setattr(torch.cuda.nvtx, "range_push", lambda name: events.append(("push", name)))
    monkeypatch.setattr(torch.cuda.nvtx, "range_pop", lambda: events.append(("pop", None)))
    x = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)  # host tensors: the call is refused before any launch
    with pytest.raises(Exception):
        fa.fwd(x, x, x)
    with pytest.raises(Exception):
        fa.bwd(x, x, x, x, torch.zeros(1, 1, 4), x)
    assert events == [("push", "fa.fwd"), ("pop", None), ("push", "fa.bwd"), ("pop", None)]


def test_off_by_default(monkeypatch):
    events = []
    monkeypatch.setattr(api, "NVTX", False)
    monkeypatch.setattr(torch.cuda.nvtx, "range_push", lambda name: events.append(name))
    x = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(Exception):
        fa.fwd(x, x, x)
    assert events == []
