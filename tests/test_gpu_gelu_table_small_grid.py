"""The GELU table kernels on small tensors, through the test-hooks build in which
every vector-path tensor takes the table path (FP8Q_TEST_GELU_TABLE_MIN_ELEMS=1).

A table kernel's grid is the CTAs the tensor needs, rounded up to whole
thread-block clusters (8 CTAs below 2^25 elements for the codes alone and below
2^26 with y), so here some CTAs have no vectors to convert but still take part
in the cluster's table build; CTA 0 also converts the scalar head and tail.
Every output is compared: y with the fixed binary32 sequence (which the GPU
GELU tests hold to the float64 tolerance), the codes and the amax with the
oracle's quantize of that y.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_bf16_equal, assert_codes_equal, assert_f32_equal, check_guards, guarded
from quantize_amax_scaling_gb300 import fp8q
from quantize_amax_scaling_gb300 import workloads as W

pytestmark = pytest.mark.gpu

# vectors of 16 elements per CTA: 1024 threads x 2 (codes only), 512 x 2 (with y)
CASES = [  # (elements, offset, with y)
    (16 * 2048 + 7, 0, False),            # 1 CTA needed, grid 8 (one whole cluster)
    (16 * (2048 * 8 + 5) + 3, 3, False),  # 9 CTAs needed, grid rounded up to 16
    (16 * 100 + 9, 5, False),             # 1 CTA needed, grid 8
    (16 * 1024 + 1, 1, True),             # 1 CTA needed, grid rounded up to 8
    (16 * (1024 * 5 - 7) + 11, 2, True),  # 5 CTAs needed, grid 8
]


@pytest.mark.parametrize("n,off,with_y", CASES)
def test_gelu_table_path_rounded_grid(hooks_lib, seq_gelu, n, off, with_y):
    dev = torch.device("cuda:0")
    g = torch.Generator(device=dev)
    g.manual_seed(n)
    hbuf = (torch.randn(n + 16, generator=g, device=dev) * 3.0).to(torch.bfloat16)
    h = hbuf[off: off + n]
    qbuf, q = guarded(n, torch.uint8, dev, off)
    ybuf, y = guarded(n, torch.bfloat16, dev, off, fill=0x5A5A) if with_y else (None, None)
    am = torch.zeros(1, device=dev)
    scale = np.float32(0.0123)
    sc = torch.full((1,), float(scale), device=dev)
    st = torch.cuda.current_stream().cuda_stream
    status = hooks_lib.fp8q_gelu_quantize_amax(h.data_ptr(), y.data_ptr() if with_y else None, q.data_ptr(), n,
                                               fp8q.E4M3FN, sc.data_ptr(), am.data_ptr(), st)
    assert status == 0
    torch.cuda.synchronize()
    hb = W.bf16_bits(h)
    want_y = seq_gelu(hb)
    rq, ra = oracle.quantize_amax(want_y, fp8q.E4M3FN, scale)
    assert_codes_equal(q.cpu().numpy(), rq, fp8q.E4M3FN, f"table q n={n}")
    assert_f32_equal([float(am)], [ra], f"table amax n={n}")
    check_guards(qbuf, n, off)
    if with_y:
        assert_bf16_equal(W.bf16_bits(y), want_y, f"table y n={n}")
        check_guards(ybuf, n, off, fill=0x5A5A)


RANDOM_CASES = 16


@pytest.mark.parametrize("k", range(RANDOM_CASES))
def test_gelu_table_path_random_small_tensors(hooks_lib, seq_gelu, k):
    """Seeded random sizes, offsets, formats, scales (the slow-path ones too) and input
    kinds through the table kernels of the test-hooks build: many threads have few or no
    elements, so the codes-alone kernel's amax often comes from its re-read."""
    rng = np.random.default_rng(1000 + k)
    dev = torch.device("cuda:0")
    n = int(rng.integers(1, 200_000))
    off = int(rng.integers(0, 16))
    with_y = bool(k % 2)
    fmt = fp8q.E4M3FN if k % 4 < 2 else fp8q.E5M2
    scale = np.float32([0.0123, 1.0, 3.7e-3, 2.0 ** 70, 0.0, 2.5e-2][k % 6])
    kind = k % 4
    v = rng.standard_normal(n + 16) * 3.0
    if kind == 1:
        v = -np.abs(v)                     # every input negative
    elif kind == 2:
        v = np.abs(v) * 0.05               # every input below about 0.3
    hb = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    if kind == 3 and n > 10:
        hb[off + int(rng.integers(0, n))] = 0x7F80 if k % 8 == 3 else 0xFFC3
    hbuf = torch.from_numpy(hb.view(np.int16).copy()).view(torch.bfloat16).to(dev)
    h = hbuf[off: off + n]
    qbuf, q = guarded(n, torch.uint8, dev, off)
    ybuf, y = guarded(n, torch.bfloat16, dev, off, fill=0x5A5A) if with_y else (None, None)
    amax0 = float(rng.choice([0.0, 0.01]))
    am = torch.full((1,), amax0, device=dev)
    sc = torch.full((1,), float(scale), device=dev)
    st = torch.cuda.current_stream().cuda_stream
    status = hooks_lib.fp8q_gelu_quantize_amax(h.data_ptr(), y.data_ptr() if with_y else None, q.data_ptr(), n,
                                               fmt, sc.data_ptr(), am.data_ptr(), st)
    assert status == 0
    torch.cuda.synchronize()
    want_y = seq_gelu(W.bf16_bits(h))
    rq, ra = oracle.quantize_amax(want_y, fmt, scale, amax0)
    what = f"case {k}: n={n} off={off} y={with_y} scale={scale}"
    assert_codes_equal(q.cpu().numpy(), rq, fmt, what + " codes")
    assert_f32_equal([float(am)], [ra], what + " amax")
    check_guards(qbuf, n, off)
    if with_y:
        assert_bf16_equal(W.bf16_bits(y), want_y, what + " y")
        check_guards(ybuf, n, off, fill=0x5A5A)


@pytest.mark.parametrize("max_cluster,with_y", [(4, False), (2, False), (4, True), (2, True)])
def test_gelu_table_falls_back_where_clusters_do_not_fit(hooks_lib, seq_gelu, max_cluster, with_y):
    """Where no cluster of a table kernel's size fits, the call takes a smaller cluster
    (clusters of 4 instead of 8) or else the direct kernel, with the same results: here the
    test build makes clusters above `max_cluster` count as not fitting."""
    dev = torch.device("cuda:0")
    n, off = 16 * 5000 + 9, 3
    g = torch.Generator(device=dev)
    g.manual_seed(max_cluster * 10 + with_y)
    hbuf = (torch.randn(n + 16, generator=g, device=dev) * 3.0).to(torch.bfloat16)
    h = hbuf[off: off + n]
    qbuf, q = guarded(n, torch.uint8, dev, off)
    ybuf, y = guarded(n, torch.bfloat16, dev, off, fill=0x5A5A) if with_y else (None, None)  # aligned like h
    am = torch.zeros(1, device=dev)
    scale = np.float32(0.0123)
    sc = torch.full((1,), float(scale), device=dev)
    st = torch.cuda.current_stream().cuda_stream
    hooks_lib.fp8q_test_set_gelu_max_cluster(max_cluster)
    try:
        status = hooks_lib.fp8q_gelu_quantize_amax(h.data_ptr(), y.data_ptr() if with_y else None, q.data_ptr(),
                                                   n, fp8q.E4M3FN, sc.data_ptr(), am.data_ptr(), st)
        torch.cuda.synchronize()
    finally:
        hooks_lib.fp8q_test_set_gelu_max_cluster(0)
    assert status == 0
    want_y = seq_gelu(W.bf16_bits(h))
    rq, ra = oracle.quantize_amax(want_y, fp8q.E4M3FN, scale)
    assert_codes_equal(q.cpu().numpy(), rq, fp8q.E4M3FN, "fallback codes")
    assert_f32_equal([float(am)], [ra], "fallback amax")
    check_guards(qbuf, n, off)
    if with_y:
        assert_bf16_equal(W.bf16_bits(y), want_y, "fallback y")
        check_guards(ybuf, n, off, fill=0x5A5A)
