"""Calls captured in a CUDA graph and replayed: every replay must compute the
product of the operands' current contents.

A stream-K launch hands partial tiles between clusters through flags that
carry the launch's epoch; a replayed graph carries the epoch it was captured
with, so the owners must clear the flags they consume.  Each replay here
changes the operands first and compares C bit for bit with an ordinary call
(same plan, same order of every sum).
"""
from __future__ import annotations

import numpy as np
import pytest

from dense_tensor_core_bf16_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.timeout(900)]

SEED = inputs.DEFAULT_SEED + 500


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tensor_core_bf16_gb300 as g
    g.lib()
    yield
    st, where = g.gemm_get_device_status(None)
    assert st == 0, f"device fault word {where:#x}"


def _bf16(bits: np.ndarray):
    return torch.from_numpy(np.array(bits, dtype=np.uint16).view(np.int16)).cuda().view(torch.bfloat16)


def _operands(M, N, K, seed):
    A, Bt = inputs.workload_operands(M, N, K, dist="normal", scaled=True, seed=seed)
    return _bf16(A), _bf16(Bt)


CASES = [
    # (M, N, K, options, what the plan must use)
    (2048, 2048, 2048, {"force_stream_k": True}, "stream_k"),   # 64 pair tiles < 76 clusters: all spread
    (4096, 4096, 1024, {"force_stream_k": True}, "stream_k"),   # a tail of 104 tiles behind 152 whole ones
    (128, 256, 16384, {"split_k": 16}, "split_k"),              # partial slices and the combine kernel
    (2048, 2048, 1024, {"force_stream_k": True, "beta": 1.0, "activation": "gelu"}, "stream_k"),  # reads C
]


@pytest.mark.parametrize("case", CASES, ids=["sk_all", "sk_tail", "splitk", "epilogue"])
def test_graph_replays_follow_the_operands(case):
    import dense_tensor_core_bf16_gb300 as g
    M, N, K, opts, uses = case
    A, Bt = _operands(M, N, K, SEED)
    st, plan = g.gemm_plan(M, N, K, g.GEMM_ROW_MAJOR, g.GEMM_COL_MAJOR, g.GEMM_OUT_F32,
                           g.options(split_k=opts.get("split_k", 0), no_stream_k=-1 if opts.get("force_stream_k") else 0))
    assert st == 0
    if uses == "stream_k":
        assert plan.stream_k_tiles > 0, "the case must exercise the stream-K hand-off"
    else:
        assert plan.split_k > 1
    if plan.workspace_bytes:
        assert g.gemm_reserve_workspace(plan.workspace_bytes) == 0
    C0 = torch.randn(M, N, device="cuda")
    C = C0.clone()
    g.matmul(A, Bt.t(), out=C, **opts)     # first call outside the capture: kernels, flags, workspace
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            g.matmul(A, Bt.t(), out=C, **opts)
    torch.cuda.synchronize()

    for r in range(4):
        A2, Bt2 = _operands(M, N, K, SEED + 1 + r)
        A.copy_(A2)
        Bt.copy_(Bt2)
        C.copy_(C0)
        graph.replay()
        torch.cuda.synchronize()
        ref = C0.clone()
        g.matmul(A, Bt.t(), out=ref, **opts)
        torch.cuda.synchronize()
        assert torch.equal(C, ref), f"replay {r} differs from an ordinary call"
