"""The benchmark step captured as a CUDA graph with parallel branches gives the oracle's results.

bench.py replays the delayed-scaling step from CUDA graphs in which quantize,
multi-tensor quantize and dequantize run on three branches forked after the amax
reset and joined before the scale update that reads their amaxes.  If the join
were missing, the update would read a partial amax; the step results after
several replays must equal the oracle's, step by step.
"""
import types

import numpy as np
import pytest
import torch

import oracle
from quantize_amax_scaling_gb300 import fp8q
from quantize_amax_scaling_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_branched_step_graph_matches_oracle():
    import bench
    dev = torch.device("cuda:0")
    H = 16
    act = W.mlp_activation(13, dev, (96, 3000)).reshape(-1)
    w1 = W.truncated_normal_weight((64, 2001), 2001, 14, dev).reshape(-1)
    w2 = W.truncated_normal_weight((2001, 64), 2001, 15, dev).reshape(-1)
    grad_q = torch.from_numpy(np.random.default_rng(16).integers(0, 256, 300001, dtype=np.uint8)).to(dev)
    hist, new, scale, scale_inv, sf = W.scale_update_inputs(dev, history_len=H)
    st = types.SimpleNamespace(fp8q=fp8q, dev=dev, act=act, w=[w1, w2], grad_q=grad_q, hist=hist,
                               amax_new=new, scale=scale, scale_inv=scale_inv, slot_format=sf,
                               q_act=torch.empty(act.numel(), dtype=torch.uint8, device=dev),
                               q_w=[torch.empty(w.numel(), dtype=torch.uint8, device=dev) for w in (w1, w2)],
                               y_grad=torch.empty(grad_q.numel(), dtype=torch.bfloat16, device=dev))

    rh, rs, ri = hist.cpu().numpy().copy(), scale.cpu().numpy().copy(), scale_inv.cpu().numpy().copy()
    ra = new.cpu().numpy().copy()
    xa, x1, x2 = W.bf16_bits(act), W.bf16_bits(w1), W.bf16_bits(w2)
    gq = grad_q.cpu().numpy()
    sfn = sf.cpu().numpy()

    def oracle_step():
        sc = rs.copy()
        qa, ra[0] = oracle.quantize_amax(xa, oracle.E4M3FN, sc[0])
        (q1, q2), (ra[1], ra[2]) = oracle.multi_quantize_amax([x1, x2], oracle.E4M3FN, [sc[1], sc[2]])
        yg = oracle.dequantize(gq, oracle.E5M2, sc[4])
        oracle.amax_scale_update(rh, ra, rs, ri, oracle.E4M3FN, oracle.ALGO_MAX, 0, sfn)
        return qa, q1, q2, yg

    stream = torch.cuda.Stream(dev)
    side = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            bench.Step.run_branched(st, stream, side)
    torch.cuda.synchronize(dev)   # capture runs nothing: the state is still the initial one

    for _ in range(3):
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize(dev)
        qa, q1, q2, yg = oracle_step()
        assert np.array_equal(st.q_act.cpu().numpy(), qa)
        assert np.array_equal(st.q_w[0].cpu().numpy(), q1)
        assert np.array_equal(st.q_w[1].cpu().numpy(), q2)
        got_y = st.y_grad.view(torch.int16).cpu().numpy().view(np.uint16)
        nan = ((yg & 0x7F80) == 0x7F80) & ((yg & 0x7F) != 0)
        assert np.array_equal(got_y[~nan], yg[~nan])
        assert np.array_equal(new.cpu().numpy(), ra)
        assert np.array_equal(hist.cpu().numpy(), rh)
        assert np.array_equal(scale.cpu().numpy(), rs)
        assert np.array_equal(scale_inv.cpu().numpy(), ri)
