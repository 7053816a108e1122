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
