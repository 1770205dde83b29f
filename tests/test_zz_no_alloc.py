"""moe_dispatch_noalloc: the dispatch entry point for callers that may not allocate device
memory (for example code inside another framework's memory pool, or a plugin host that hands
over only the tensors it owns).  It keeps its scratch in a fixed array inside the library
instead of a caller workspace.  These checks run it through the C ABI, twice in a row with
different shapes (the array is shared and keeps the previous call's contents), and require its
outputs to equal those of moe_dispatch bit for bit, as every dispatch output is an integer or a
copied row."""
import numpy as np
import pytest
import torch

import moe_inputs
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _outputs(T, E, k, d):
    i32 = dict(dtype=torch.int32, device=DEV)
    return {"counts": torch.full((E,), -9, **i32), "kept": torch.full((E,), -9, **i32),
            "offsets": torch.full((E + 1,), -9, **i32), "pos": torch.full((T, k), -9, **i32),
            "row_of": torch.full((T, k), -9, **i32), "perm": torch.full((T * k,), -9, **i32),
            "x_perm": torch.zeros((T * k, d), dtype=torch.bfloat16, device=DEV),
            "n_dropped": torch.full((1,), -9, **i32)}


def _route(m, wl, cfg, inp):
    ws = m.workspace(cfg)
    logits = torch.empty((wl.T, wl.E), dtype=torch.float32, device=DEV)
    idx = torch.empty((wl.T, wl.k), dtype=torch.int32, device=DEV)
    w = torch.empty((wl.T, wl.k), dtype=torch.float32, device=DEV)
    m.moe_router_topk(cfg, inp["x"], inp["w_gate"], inp["bias"], logits, idx, w, ws)
    return idx, ws


def _check_case(m, wl, gather=True):
    """Both dispatch entry points on the same routed indices; gather=False passes no x and no
    x_perm (counts, positions and permutation only)."""
    cfg = U.config_of(wl)
    inp = moe_inputs.make_router_inputs(wl, device=DEV)
    idx, ws = _route(m, wl, cfg, inp)
    a = _outputs(wl.T, wl.E, wl.k, wl.d)
    b = _outputs(wl.T, wl.E, wl.k, wl.d)
    names = ["counts", "kept", "offsets", "pos", "row_of", "perm"]
    x = inp["x"] if gather else None
    m.moe_dispatch(cfg, idx, x, *[a[n] for n in names], a["x_perm"] if gather else None,
                   a["n_dropped"], ws)
    status = torch.full((2,), 123, dtype=torch.int32, device=DEV)
    m.moe_dispatch_noalloc(cfg, idx, x, *[b[n] for n in names], b["x_perm"] if gather else None,
                           b["n_dropped"], status)
    torch.cuda.synchronize()
    assert m.sync_status(ws) == 0
    assert status.tolist() == [0, 0]
    for n in names + ["n_dropped"]:
        assert torch.equal(a[n], b[n]), n
    nk = int(a["offsets"][-1].item())
    if gather:
        assert torch.equal(a["x_perm"][:nk], b["x_perm"][:nk])
    else:
        assert not b["x_perm"].any()      # no rows were gathered
    return int(a["n_dropped"].item())


def test_noalloc_dispatch_equals_workspace_dispatch_in_a_row():
    m = U.lib()
    first = moe_inputs.workload("v3", T=700, d=256, E=64, F=256, F_shared=256,
                                capacity_factor=1.25)
    second = moe_inputs.workload("mixtral_collapsed", T=1000, d=256, F=256, capacity_factor=1.0)
    # T <= 256 runs the one-launch dispatch, which uses only the array's M-tile-prefix words
    third = moe_inputs.workload("mixtral", T=200, d=256, E=8, k=2, F=256, capacity_factor=1.0)
    d1 = _check_case(m, first)
    d2 = _check_case(m, second)        # same scratch array, different shape, right after
    d3 = _check_case(m, third)
    d4 = _check_case(m, second, gather=False)
    assert d1 > 0 and d2 > 0 and d3 > 0 and d4 == d2


def test_noalloc_dispatch_refuses_more_than_its_scratch_holds():
    m = U.lib()
    cfg = m.make_config(65537, 128, 8, 2, 128)
    fake = torch.zeros(1, dtype=torch.int32, device=DEV)
    with pytest.raises(m.MoeError) as err:
        m.moe_dispatch_noalloc(cfg, fake, None, fake, fake, fake, fake, fake, fake, None, fake,
                               fake)
    assert err.value.status == -2
