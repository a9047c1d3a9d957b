"""A MuonH step captured into a CUDA graph and replayed equals the eager
step, bit for bit.

The step of a several-bucket set forks independent buckets onto the
library's side streams and joins them back with events; under stream
capture those streams join the capture through the same events, so the
whole step (small-matrix kernel, momentum, Newton-Schulz GEMMs, hyperball)
becomes one graph.  The graph is replayed twice with new gradients copied
into its static buffers; each replay must equal an eager step from the same
state.  One eager step first builds the plan, the side streams and the
event pool, so nothing is created while capturing.
"""

import numpy as np
import pytest
import torch

import muonh_workloads as wl

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import hyperball_constrained_muon_muonh_b300 as mh

# buckets on several streams, a small-matrix group and an fp32 (s <= 80) one
SHAPES = [(512, 512)] * 2 + [(384, 1024)] * 3 + [(1024, 384)] * 2 + [(256, 128)] * 2 + [(77, 77)]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mh.get_status()
    yield
    assert mh.get_status() & mh.STATUS_KERNEL_TIMEOUT == 0


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int32).numpy()


@pytest.mark.parametrize("optimizer", ["muonh", "muon"])
def test_step_replayed_from_cuda_graph_equals_eager(optimizer):
    work = wl.ragged(SHAPES)

    def make():
        ws = work.weights("cuda")
        if optimizer == "muonh":
            opt = mh.MuonH(ws, lr=work.lr, beta=work.beta, ns_steps=work.ns_steps, ns_coeffs=work.coeffs,
                           eps=work.eps, bf16_copies=True)
        else:
            opt = mh.Muon(ws, lr=work.lr, beta=work.beta, weight_decay=0.1, ns_steps=work.ns_steps,
                          ns_coeffs=work.coeffs, eps=work.eps, bf16_copies=True)
        return ws, opt

    ws_e, opt_e = make()
    ws_g, opt_g = make()
    static = [g.clone() for g in work.grads(0, "cuda")]
    # eager step 0 on both (plan, side streams, events, cached matrix array)
    opt_e.step(work.grads(0, "cuda"))
    opt_g.step(static)
    torch.cuda.synchronize()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        opt_g.step(static)
    torch.cuda.synchronize()

    for t in (1, 2):
        gs = work.grads(t, "cuda")
        for dst, src in zip(static, gs):
            dst.copy_(src)
        graph.replay()
        opt_e.step(gs)
        torch.cuda.synchronize()
        assert mh.get_status() == 0
        for k in range(len(SHAPES)):
            assert np.array_equal(_bits(ws_g[k]), _bits(ws_e[k])), f"step {t}, W of matrix {k} {SHAPES[k]}"
            assert np.array_equal(_bits(opt_g.moms[k]), _bits(opt_e.moms[k])), f"step {t}, M of matrix {k}"
            assert np.array_equal(opt_g.bf16[k].detach().cpu().view(torch.int16).numpy(),
                                  opt_e.bf16[k].detach().cpu().view(torch.int16).numpy()), f"step {t}, bf16 {k}"
