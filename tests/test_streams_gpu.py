"""Calls on different streams with their own workspaces do not interfere.

The C ABI keeps every piece of per-call device state (split partials, arrival
tickets, selection scores, first-digit histograms, the status word) in the
caller's workspace, so two decode steps that share nothing but the library
may run at the same time on two streams.  Each result must then be bit for
bit the one the step gives alone (the kernels are deterministic: the split
merge reads the partials in a fixed order whichever CTA arrives last).
"""
import pytest
import torch

import sparse_attention_td_gb300 as td
import workloads as W

pytestmark = pytest.mark.gpu
D = 128
MODES = [W.FULL, W.FULL_SELECT, W.SPARSE, W.SPARSE, W.FULL_SELECT, W.SPARSE]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _case(seed, B, Hq, Hkv, N, k):
    """One step's inputs and outputs: grouped-query (tensor-core kernels) or
    MHA (CUDA-core kernels), ragged lengths."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    L = len(MODES)

    def rnd(*shape):
        return torch.randn(*shape, generator=g, device="cuda").to(torch.bfloat16)

    c = {
        "shape": td.make_shape(B, Hq, Hkv, N, scale=td.default_scale(D)),
        "q": [rnd(B, Hq, D) for _ in range(L)],
        "K": [rnd(B, Hkv, N, D) for _ in range(L)],
        "V": [rnd(B, Hkv, N, D) for _ in range(L)],
        "seq": torch.tensor([N - 37 * b for b in range(B)], dtype=torch.int32, device="cuda"),
        "k": k,
        "outs": [torch.zeros(B, Hq, D, dtype=torch.bfloat16, device="cuda") for _ in range(L)],
        "outs32": [torch.zeros(B, Hq, D, dtype=torch.float32, device="cuda") for _ in range(L)],
        "idx": torch.full((B, Hkv, k), -1, dtype=torch.int32, device="cuda"),
    }
    c["ws"] = td.Workspace(c["shape"], k)
    return c


def _step(c, stream=None):
    td.td_decode_step(c["shape"], MODES, c["q"], c["K"], c["V"], c["seq"], c["k"], c["idx"],
                      c["outs"], c["outs32"], c["ws"], stream=stream)


def _snapshot(c):
    return [c["idx"].clone()] + [o.clone() for o in c["outs"]] + [o.clone() for o in c["outs32"]]


def _clear(c):
    for o in c["outs"] + c["outs32"]:
        o.zero_()
    c["idx"].fill_(-1)


def _cases():
    return [_case(11, 2, 16, 4, 9000, 256),    # G = 4: tensor-core kernels
            _case(12, 1, 16, 16, 7000, 300)]   # G = 1: CUDA-core kernels


def test_concurrent_steps_on_two_streams_match_each_alone():
    cases = _cases()
    alone = []
    for c in cases:
        _step(c)
        torch.cuda.synchronize()
        alone.append(_snapshot(c))
        _clear(c)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for it in range(8):                       # both orders of launch, many overlaps
        order = (0, 1) if it % 2 == 0 else (1, 0)
        for i in order:
            _step(cases[i], stream=streams[i])
    torch.cuda.synchronize()
    for c, ref in zip(cases, alone):
        assert c["ws"].status() == 0
        for a, b in zip(_snapshot(c), ref):
            assert torch.equal(a, b)


def test_concurrent_plans_on_two_streams_match_each_alone():
    cases = _cases()
    alone = []
    for c in cases:
        _step(c)
        torch.cuda.synchronize()
        alone.append(_snapshot(c))
        _clear(c)
    torch.cuda.synchronize()
    plans = [td.Plan(c["shape"], MODES, c["q"], c["K"], c["V"], c["seq"], c["k"], c["idx"],
                     c["outs"], c["outs32"], c["ws"]) for c in cases]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for _ in range(8):
        for p, s in zip(plans, streams):
            p.launch(stream=s)
    torch.cuda.synchronize()
    for p in plans:
        p.close()
    for c, ref in zip(cases, alone):
        assert c["ws"].status() == 0
        for a, b in zip(_snapshot(c), ref):
            assert torch.equal(a, b)
