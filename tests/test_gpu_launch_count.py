"""Each entry point is one kernel launch.

Each call is captured into a CUDA graph and the graph's nodes are counted
through the driver API: a call that launched two kernels, or a kernel plus
a memset, would show up as more than one node.
"""
import ctypes
import os

import pytest
import torch

from conftest import ROOT
from quantize_amax_scaling_gb300 import fp8q
from quantize_amax_scaling_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CU_GRAPH_NODE_TYPE_KERNEL = 0


def _graph_nodes(fn, stream):
    """(kernel nodes, all nodes) of a graph that captured fn() on `stream`."""
    drv = ctypes.CDLL("libcuda.so.1")
    g = torch.cuda.CUDAGraph(keep_graph=True)
    with torch.cuda.graph(g, stream=stream):
        fn()
    handle = ctypes.c_void_p(g.raw_cuda_graph())
    n = ctypes.c_size_t(0)
    assert drv.cuGraphGetNodes(handle, None, ctypes.byref(n)) == 0
    nodes = (ctypes.c_void_p * max(1, n.value))()
    assert drv.cuGraphGetNodes(handle, nodes, ctypes.byref(n)) == 0
    kernels = 0
    for i in range(n.value):
        t = ctypes.c_int(-1)
        assert drv.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) == 0
        kernels += t.value == CU_GRAPH_NODE_TYPE_KERNEL
    del g
    return kernels, n.value


def test_every_entry_point_is_one_launch():
    dev = torch.device("cuda:0")
    s = torch.cuda.Stream()
    x = W.mlp_activation(1, dev, (256, 4096)).reshape(-1)
    q = torch.empty(x.numel(), dtype=torch.uint8, device=dev)
    y = torch.empty(x.numel(), dtype=torch.bfloat16, device=dev)
    sc = torch.full((4,), 0.05, device=dev)
    am = torch.zeros(4, device=dev)
    hist, new, scale, scale_inv, sf = W.scale_update_inputs(dev)
    head = torch.full((new.numel(),), 1023, dtype=torch.int32, device=dev)
    lg, lb = W.layernorm_params(4096, device=dev)
    head2 = torch.empty_like(head)
    xl = W.mlp_activation(2, dev, (4096, 4096)).reshape(-1)   # 2^24 elements: the GELU table path
    ql = torch.empty(xl.numel(), dtype=torch.uint8, device=dev)
    xt = W.mlp_activation(3, dev, (3000, 16384)).reshape(-1)  # 3000 tiles: one CTA per tile
    qt = torch.empty(xt.numel(), dtype=torch.uint8, device=dev)
    third = x.numel() // 3
    ws, qs = [x[:third], x[third:]], [q[:third], q[third:]]
    st = s.cuda_stream
    calls = {
        "quantize, persistent grid": lambda: fp8q.fp8q_quantize_amax(x, q, fp8q.E4M3FN, sc[0:1], am[0:1], st),
        "quantize, one CTA per tile": lambda: fp8q.fp8q_quantize_amax(xt, qt, fp8q.E4M3FN, sc[0:1], am[0:1], st),
        "multi (2 tensors)": lambda: fp8q.fp8q_multi_quantize_amax(ws, qs, fp8q.E4M3FN, [sc[1:2], sc[2:3]],
                                                                   [am[1:2], am[2:3]], st),
        "dequantize": lambda: fp8q.fp8q_dequantize(q, y, fp8q.E4M3FN, sc[0:1], st),
        "update, 576 slots": lambda: fp8q.fp8q_amax_scale_update(hist, new, scale, scale_inv, fp8q.E4M3FN,
                                                                 fp8q.ALGO_MAX, 0, sf, st),
        "ring update, 576 slots": lambda: fp8q.fp8q_amax_scale_update_ring(hist, head, new, scale, scale_inv,
                                                                           fp8q.E4M3FN, fp8q.ALGO_MAX, 0, sf,
                                                                           st),
        "fused Q->DQ": lambda: fp8q.fp8q_qdq_amax(x, y, fp8q.E4M3FN, sc[3:4], am[3:4], st),
        "GELU + quantize": lambda: fp8q.fp8q_gelu_quantize_amax(x, y, q, fp8q.E4M3FN, sc[0:1], am[0:1], st),
        "GELU + quantize, table path": lambda: fp8q.fp8q_gelu_quantize_amax(xl, None, ql, fp8q.E4M3FN, sc[0:1],
                                                                          am[0:1], st),
        "ring update + quantize": lambda: fp8q.fp8q_amax_scale_update_ring_quantize(hist, head, head2, new, scale,
                                                                                     scale_inv, x, q, 7, am[2:3],
                                                                                     fp8q.E4M3FN, fp8q.ALGO_MAX,
                                                                                     0, sf, stream=st),
        "LayerNorm + quantize": lambda: fp8q.fp8q_layernorm_quantize_amax(x.view(256, 4096), y.view(256, 4096),
                                                                         q.view(256, 4096), lg, lb, fp8q.E4M3FN,
                                                                         sc[1:2], am[1:2], stream=st),
    }
    with torch.cuda.stream(s):
        for fn in calls.values():
            fn()                               # first calls outside capture
    s.synchronize()
    for name, fn in calls.items():
        kernels, nodes = _graph_nodes(fn, s)
        assert (kernels, nodes) == (1, 1), (name, kernels, nodes)


@pytest.mark.gpu
def test_layernorm_first_call_inside_graph_capture():
    """The first use on a device of the calls that query the device (the LayerNorm call:
    function attribute and occupancy; the quantize of a mid-size tensor: the SM count) may
    itself be captured: in a fresh process, capture them, replay, and compare with eager
    calls."""
    import subprocess
    import sys
    code = r'''
import torch
from quantize_amax_scaling_gb300 import fp8q, workloads as W
dev = torch.device("cuda:0")
x = W.residual_stream(seed=1, device=dev, shape=(64, 4096))
g, b = W.layernorm_params(4096, device=dev)
sc = torch.full((1,), 0.02, device=dev)
q, am = torch.empty(x.shape, dtype=torch.uint8, device=dev), torch.zeros(1, device=dev)
xm = W.mlp_activation(5, dev, (512, 4096)).reshape(-1)
qm, amm = torch.empty(xm.numel(), dtype=torch.uint8, device=dev), torch.zeros(1, device=dev)
gr = torch.cuda.CUDAGraph()
with torch.cuda.graph(gr, stream=torch.cuda.Stream()):
    fp8q.fp8q_layernorm_quantize_amax(x, None, q, g, b, fp8q.E4M3FN, sc, am)
    fp8q.fp8q_quantize_amax(xm, qm, fp8q.E4M3FN, sc, amm)
gr.replay()
torch.cuda.synchronize()
q2, am2 = torch.empty_like(q), torch.zeros(1, device=dev)
fp8q.fp8q_layernorm_quantize_amax(x, None, q2, g, b, fp8q.E4M3FN, sc, am2)
qm2, amm2 = torch.empty_like(qm), torch.zeros(1, device=dev)
fp8q.fp8q_quantize_amax(xm, qm2, fp8q.E4M3FN, sc, amm2)
torch.cuda.synchronize()
assert torch.equal(q, q2) and float(am) == float(am2)
assert torch.equal(qm, qm2) and float(amm) == float(amm2)
print("OK")
'''
    env = dict(os.environ, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout + r.stderr


def test_cluster_kernels_first_call_inside_graph_capture():
    """The same for the calls that launch thread-block clusters and query how many fit
    (cudaOccupancyMaxActiveClusters) on their first use: the LayerNorm on rows of 12288
    and the two GELU table kernels."""
    import subprocess
    import sys
    code = r'''
import torch
from quantize_amax_scaling_gb300 import fp8q, workloads as W
dev = torch.device("cuda:0")
x = W.residual_stream(seed=2, device=dev, shape=(40, 12288))
g, b = W.layernorm_params(12288, device=dev)
sc = torch.full((1,), 0.02, device=dev)
q, am = torch.empty(x.shape, dtype=torch.uint8, device=dev), torch.zeros(1, device=dev)
gen = torch.Generator(device=dev); gen.manual_seed(3)
h = torch.randn(1 << 25, generator=gen, device=dev).to(torch.bfloat16)
gy, gq, gam = torch.empty_like(h), torch.empty(h.numel(), dtype=torch.uint8, device=dev), torch.zeros(1, device=dev)
hq, hqam = torch.empty(1 << 23, dtype=torch.uint8, device=dev), torch.zeros(1, device=dev)
gr = torch.cuda.CUDAGraph()
with torch.cuda.graph(gr, stream=torch.cuda.Stream()):
    fp8q.fp8q_layernorm_quantize_amax(x, None, q, g, b, fp8q.E4M3FN, sc, am)
    fp8q.fp8q_gelu_quantize_amax(h, gy, gq, fp8q.E4M3FN, sc, gam)
    fp8q.fp8q_gelu_quantize_amax(h[: 1 << 23], None, hq, fp8q.E4M3FN, sc, hqam)
gr.replay()
torch.cuda.synchronize()
q2, am2 = torch.empty_like(q), torch.zeros(1, device=dev)
fp8q.fp8q_layernorm_quantize_amax(x, None, q2, g, b, fp8q.E4M3FN, sc, am2)
gy2, gq2, gam2 = torch.empty_like(gy), torch.empty_like(gq), torch.zeros(1, device=dev)
fp8q.fp8q_gelu_quantize_amax(h, gy2, gq2, fp8q.E4M3FN, sc, gam2)
hq2, hqam2 = torch.empty_like(hq), torch.zeros(1, device=dev)
fp8q.fp8q_gelu_quantize_amax(h[: 1 << 23], None, hq2, fp8q.E4M3FN, sc, hqam2)
torch.cuda.synchronize()
assert torch.equal(q, q2) and float(am) == float(am2)
assert torch.equal(gy.view(torch.int16), gy2.view(torch.int16)) and torch.equal(gq, gq2) and float(gam) == float(gam2)
assert torch.equal(hq, hq2) and float(hqam) == float(hqam2)
print("OK")
'''
    env = dict(os.environ, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout + r.stderr
