"""Failure detection on the GPU without a fault: a bounded wait that nothing
satisfies runs out, the kernel records MOE_ERR_DEVICE_TIMEOUT in the
workspace status word and returns, and the context stays usable."""
import time

import pytest
import torch

import moe_inputs as mi
import oracle
import mixture_experts_ffn_permute_gb300 as moe
from mixture_experts_ffn_permute_gb300 import _build
from parity import assert_bf16_close, assert_equal

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    moe.load()


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    shape = mi.TINY
    p = moe.Problem.make(shape.T, shape.H, shape.F, shape.E, shape.k)
    ws = moe.alloc_workspace(p)
    moe.clear_device_status(ws)
    limit = 100_000_000  # 0.1 s
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    moe.selftest_wait_timeout(ws, limit)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert moe.STATUS_NAMES[moe.get_device_status(ws)] == "MOE_ERR_DEVICE_TIMEOUT"
    assert dt >= 0.09, dt

    # the same context and workspace still run the layer correctly
    moe.clear_device_status(ws)
    inp = mi.make_inputs(shape, seed=0)
    ref = oracle.moe_forward(inp["x"], inp["logits"], inp["w1"], inp["w2"], shape.k)
    d = {k: v.to(DEV) for k, v in inp.items()}
    out = torch.empty(shape.T, shape.H, dtype=torch.bfloat16, device=DEV)
    idx = torch.empty(shape.T, shape.k, dtype=torch.int32, device=DEV)
    moe.forward(p, d["x"], d["logits"], d["w1"], d["w2"], out, ws, idx)
    assert moe.get_device_status(ws) == 0
    assert_equal(idx, ref["topk_idx"], "topk_idx")
    assert_bf16_close(out, ref["out"], "out after the timeout self-test")
