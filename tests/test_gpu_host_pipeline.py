"""The end-to-end measurement's piecewise host pipeline gives the oracle's results.

bench.py times the step from pinned host memory back to pinned host memory
with tensors cut into pieces on three streams; the path is elementwise and amax
is max-accumulated, so the host results must equal whole-tensor results.
"""
import types

import numpy as np
import pytest
import torch

import oracle
from quantize_amax_scaling_gb300 import fp8q
from quantize_amax_scaling_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_piecewise_host_pipeline_matches_oracle(monkeypatch):
    import bench
    dev = torch.device("cuda:0")
    S, H = 576, 16
    act = W.mlp_activation(3, dev, (96, 1000)).reshape(-1)
    w1 = W.truncated_normal_weight((40, 1001), 1001, 4, dev).reshape(-1)
    w2 = W.truncated_normal_weight((1001, 40), 1001, 5, dev).reshape(-1)
    grad_q = torch.from_numpy(np.random.default_rng(6).integers(0, 256, 77777, dtype=np.uint8)).to(dev)
    hist, new, scale, scale_inv, sf = W.scale_update_inputs(dev, history_len=H)
    st = types.SimpleNamespace(fp8q=fp8q, dev=dev, act=act, w=[w1, w2], grad_q=grad_q, hist=hist,
                               amax_new=new, scale=scale, scale_inv=scale_inv, slot_format=sf,
                               q_act=torch.empty(act.numel(), dtype=torch.uint8, device=dev),
                               q_w=[torch.empty(w.numel(), dtype=torch.uint8, device=dev) for w in (w1, w2)],
                               y_grad=torch.empty(grad_q.numel(), dtype=torch.bfloat16, device=dev))
    host_in = {"act": act.cpu().pin_memory(), "w1": w1.cpu().pin_memory(), "w2": w2.cpu().pin_memory(),
               "grad_q": grad_q.cpu().pin_memory(), "amax_new": new.cpu().pin_memory()}
    host_out = {"q_act": torch.empty(act.numel(), dtype=torch.uint8).pin_memory(),
                "q_w1": torch.empty(w1.numel(), dtype=torch.uint8).pin_memory(),
                "q_w2": torch.empty(w2.numel(), dtype=torch.uint8).pin_memory(),
                "y_grad": torch.empty(grad_q.numel(), dtype=torch.bfloat16).pin_memory(),
                "scale": torch.empty(S).pin_memory(), "scale_inv": torch.empty(S).pin_memory()}
    monkeypatch.setattr(bench._HostPipeline, "CHUNK", 10007)      # several uneven pieces per tensor
    comp = torch.cuda.Stream()
    pipe = bench._HostPipeline(st, host_in, host_out, comp)
    assert len(pipe.pieces) > 12

    rh, rs, ri = hist.cpu().numpy().copy(), scale.cpu().numpy().copy(), scale_inv.cpu().numpy().copy()
    rnew = new.cpu().numpy().copy()
    xa, x1, x2 = W.bf16_bits(act), W.bf16_bits(w1), W.bf16_bits(w2)
    gq = grad_q.cpu().numpy()
    for _ in range(3):
        pipe.run()
        torch.cuda.synchronize()
        sc = rs.copy()
        ra = rnew.copy()
        qa, ra[0] = oracle.quantize_amax(xa, oracle.E4M3FN, sc[0])
        (q1, q2), (ra[1], ra[2]) = oracle.multi_quantize_amax([x1, x2], oracle.E4M3FN, [sc[1], sc[2]])
        yg = oracle.dequantize(gq, oracle.E5M2, sc[4])
        oracle.amax_scale_update(rh, ra, rs, ri, oracle.E4M3FN, oracle.ALGO_MAX, 0, sf.cpu().numpy())
        assert np.array_equal(host_out["q_act"].numpy(), qa)
        assert np.array_equal(host_out["q_w1"].numpy(), q1)
        assert np.array_equal(host_out["q_w2"].numpy(), q2)
        got_y = host_out["y_grad"].view(torch.int16).numpy().view(np.uint16)
        nan = ((yg & 0x7F80) == 0x7F80) & ((yg & 0x7F) != 0)
        assert np.array_equal(got_y[~nan], yg[~nan])
        assert np.array_equal(host_out["scale"].numpy(), rs)
        assert np.array_equal(host_out["scale_inv"].numpy(), ri)
