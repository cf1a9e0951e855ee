"""GPU parity of ss_ssd_chunk_scan_fwd against the fp64 oracle (C ABI, cuda:0)."""
import os

import numpy as np
import pytest
import torch

from selective_state_space_146_b300 import _abi, inputs
from tests.parity_util import check_close, cuda_inputs, oracle_ssd, oracle_ssd_units, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture
def ssd_path(request):
    old = os.environ.get("SS_SSD_PATH")
    val = getattr(request, "param", None)
    if val:
        os.environ["SS_SSD_PATH"] = val
    else:
        os.environ.pop("SS_SSD_PATH", None)
    yield val
    if old is None:
        os.environ.pop("SS_SSD_PATH", None)
    else:
        os.environ["SS_SSD_PATH"] = old


def _run(inp, dev, chunk):
    g = cuda_inputs(inp, dev)
    y, s = _abi.ssd_chunk_scan_fwd(g["x"], g["dt"], g["A_head"], g["B"], g["C"], g["D"],
                                   chunk=chunk, return_last_state=True)
    torch.cuda.synchronize()
    assert _abi.device_error() == 0
    return y, s


CASES = [
    # Bsz, L, H, P, N, G, dtype, chunk, skip
    (1, 64, 2, 4, 8, 1, "f32", 64, True),
    (2, 300, 4, 16, 32, 2, "f32", 128, True),
    (2, 256, 4, 64, 128, 1, "bf16", 64, True),
    (1, 1000, 8, 64, 128, 1, "bf16", 256, False),   # ragged last chunk
    (2, 512, 4, 64, 128, 2, "bf16", 128, True),
    (1, 1, 2, 8, 16, 1, "f32", 64, True),            # L = 1
    (1, 130, 3, 5, 7, 3, "f32", 64, True),           # odd sizes
    (1, 384, 2, 64, 256, 1, "bf16", 64, True),       # N = 256
    (1, 384, 3, 64, 128, 1, "bf16", 128, True),      # odd heads per group: one head per CTA
    (2, 200, 8, 64, 128, 4, "bf16", 128, True),      # two heads per group, ragged tail
    (1, 100, 2, 64, 128, 1, "bf16", 128, True),      # a single, partial 128-step block
    (3, 128, 2, 64, 128, 1, "bf16", 64, False),      # exactly one block
    (1, 129, 4, 64, 128, 2, "bf16", 128, True),      # a second block of one step
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:8])))
@pytest.mark.parametrize("ssd_path", [None, "general", "tc1"], indirect=True)
def test_small_shapes(cuda_device, ssd_path, case):
    Bsz, L, H, P, N, G, dt, chunk, skip = case
    inp = inputs.ssd_inputs(Bsz, L, H, P, N, G, dt, skip=skip, seed=L + H)
    y, s = _run(inp, cuda_device, chunk)
    yo, so = oracle_ssd(inp)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    check_close(to_np(y), yo, tdt, "y")
    check_close(to_np(s), so, tdt, "last_state")


def test_chunk_size_does_not_change_result(cuda_device):
    inp = inputs.ssd_inputs(1, 768, 4, 64, 128, 1, "bf16", seed=9)
    outs = [_run(inp, cuda_device, c) for c in (64, 128, 256)]
    for y, s in outs[1:]:
        check_close(to_np(y), to_np(outs[0][0]), torch.bfloat16, "y across chunk sizes")
        check_close(to_np(s), to_np(outs[0][1]), torch.bfloat16, "state across chunk sizes")


@pytest.mark.parametrize("ssd_path", [None, "tc1"], indirect=True)
def test_full_size_workload_sampled(cuda_device, ssd_path):
    cfg = inputs.WORKLOADS["mamba2_ssd"]
    inp = inputs.workload_ssd_inputs(cfg)
    y, s = _run(inp, cuda_device, cfg.chunk)
    units = inputs.sample_units(cfg.batch * cfg.nheads, 10, seed=2)
    yo, so = oracle_ssd_units(inp, units)
    yg = np.stack([to_np(y[u // cfg.nheads, :, u % cfg.nheads]) for u in units])
    sg = np.stack([to_np(s[u // cfg.nheads, u % cfg.nheads]) for u in units])
    check_close(yg, yo, torch.bfloat16, "ssd y (sampled heads)")
    check_close(sg, so, torch.bfloat16, "ssd last_state (sampled heads)")
    assert bool(torch.isfinite(y).all())
