"""cp_direct and cp_cutoff (with a caller-owned workspace) launch only
stream-ordered work with no allocation or synchronisation, so a CUDA graph
can capture them once and replay them: replays give the eager results and
follow in-place changes of the input buffers."""
import numpy as np
import pytest
import torch

import direct_coulomb_summation_gb300 as cp
import workloads
from gpu_util import to_dev

pytestmark = pytest.mark.gpu


def test_graph_capture_and_replay():
    w = workloads.random_case(71, 3000, (40, 24, 12), margin=2.0)
    c, b = 3.0, 1.0
    a = to_dev(w.atoms)
    Vd = torch.empty((12, 24, 40), device="cuda")
    Vc = torch.empty((12, 24, 40), device="cuda")
    need = cp.cutoff_workspace_bytes(w.n_atoms, w.shape, w.origin, w.h, c, b, 0)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    # eager runs (also warm the library's per-device caches before capture)
    ref_d = cp.direct(a, w.shape, w.origin, w.h).clone()
    ref_c = cp.cutoff(a, w.shape, w.origin, w.h, c, b, 0, workspace=ws).clone()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cp.direct(a, w.shape, w.origin, w.h, out=Vd)
        cp.cutoff(a, w.shape, w.origin, w.h, c, b, 0, workspace=ws, out=Vc)
    Vd.zero_()
    Vc.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(Vd, ref_d)
    assert torch.equal(Vc, ref_c)
    # the graph reads the atoms in place: doubling every charge doubles V
    a[:, 3] *= 2.0
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(Vd, 2.0 * ref_d)
    assert torch.allclose(Vc, 2.0 * ref_c, rtol=0, atol=0)
    assert cp.device_status() == 0


def test_graph_capture_of_the_multilevel_map():
    """cutoff + cp_msm_longrange (accumulating) in one graph: the replay gives
    the eager multilevel map, bit for bit."""
    w = workloads.random_case(72, 2500, (36, 20, 16), margin=3.0, cutoff=4.0, bin_size=2.0)
    h0 = 1.0
    a = to_dev(w.atoms)
    dom = cp.atom_bounds(a)
    V = torch.empty((16, 20, 36), device="cuda")
    need_c = cp.cutoff_workspace_bytes(w.n_atoms, w.shape, w.origin, w.h, w.cutoff, w.bin_size, 0)
    need_m = cp.msm_workspace_bytes(w.n_atoms, w.shape, w.origin, w.h, w.cutoff, h0, dom)
    ws_c = torch.empty(need_c, dtype=torch.uint8, device="cuda")
    ws_m = torch.empty(need_m, dtype=torch.uint8, device="cuda")

    def run(out):
        cp.cutoff(a, w.shape, w.origin, w.h, w.cutoff, w.bin_size, 0, workspace=ws_c, out=out)
        cp.msm_longrange(a, w.shape, w.origin, w.h, w.cutoff, h0, domain=dom, accumulate=True, workspace=ws_m,
                         out=out)

    ref = torch.empty_like(V)
    run(ref)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run(V)
    V.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(V, ref)
    assert cp.device_status() == 0
