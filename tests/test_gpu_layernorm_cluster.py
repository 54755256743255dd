"""LayerNorm rows longer than 4096: the kernel that splits each row over a thread-block
cluster of ceil(H / 4096) CTAs (each CTA a column slice, the partial sums exchanged over
distributed shared memory), and the single-CTA kernel the library falls back to where no
such cluster fits.

Row lengths are picked around every cluster size from 2 to 8 and around uneven last
slices; row counts make each cluster loop over several batches.  y is held to the
LayerNorm tolerance of the float64 definition on every element, and the codes and amax
are exact against the oracle's quantize of y.  The fallback runs through the library's
test-hooks build, in which clusters above a set size count as not fitting.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_codes_equal, assert_f32_equal, f32, par_quantize_amax
from quantize_amax_scaling_gb300 import fp8q
from quantize_amax_scaling_gb300 import workloads as W
from test_gpu_producers import assert_layernorm_y, check_layernorm

pytestmark = pytest.mark.gpu

E4M3FN, E5M2 = fp8q.E4M3FN, fp8q.E5M2


@pytest.fixture(scope="module")
def dev():
    fp8q.lib()
    return torch.device("cuda:0")


def cluster_size(H):
    return -(-(H // 8) // 512)


# (rows, H): cluster sizes 2 .. 8, last slices shorter than the others, many batches per cluster
CLUSTER_SHAPES = [(513, 4112), (3000, 8192), (77, 8208), (1200, 12288), (41, 12304), (600, 16384),
                  (303, 20480), (150, 24576), (128, 24592), (95, 28688), (260, 32768), (7, 5136), (1, 32752)]


def test_the_shapes_cover_every_cluster_size():
    assert sorted({cluster_size(H) for _, H in CLUSTER_SHAPES}) == [2, 3, 4, 5, 6, 7, 8]


@pytest.mark.parametrize("rows,H", CLUSTER_SHAPES)
def test_layernorm_cluster_shapes(dev, rows, H):
    x = W.residual_stream(seed=rows * 31 + H, device=dev, shape=(rows, H))
    gamma, beta = W.layernorm_params(H, seed=H + 3, device=dev)
    for k, (fmt, scale) in enumerate([(E4M3FN, 0.0123), (E5M2, 2.0 ** 70)]):
        check_layernorm(x, gamma, beta, fmt, scale, dev, amax0=0.5 * k, what=f"{rows}x{H} cluster {cluster_size(H)}")


def test_layernorm_cluster_output_is_deterministic(dev):
    """Every CTA of a cluster adds the partial sums in rank order: the same bits every call."""
    x = W.residual_stream(seed=4, device=dev, shape=(1000, 12288))
    gamma, beta = W.layernorm_params(12288, device=dev)
    outs = []
    for _ in range(3):
        y = torch.empty_like(x)
        q = torch.empty(x.shape, dtype=torch.uint8, device=dev)
        am = f32(0.0, dev)
        fp8q.fp8q_layernorm_quantize_amax(x, y, q, gamma, beta, E4M3FN, f32(0.02, dev), am)
        torch.cuda.synchronize()
        outs.append((y.view(torch.int16).clone(), q.clone(), float(am)))
    for y, q, a in outs[1:]:
        assert torch.equal(y, outs[0][0]) and torch.equal(q, outs[0][1]) and a == outs[0][2]


def _hooked_layernorm(L, x, gamma, beta, fmt, scale, dev, want_y):
    rows, H = x.shape
    y = torch.empty_like(x) if want_y else None
    q = torch.empty((rows, H), dtype=torch.uint8, device=dev)
    am = f32(0.0, dev)
    sc = f32(scale, dev)
    st = L.fp8q_layernorm_quantize_amax(x.data_ptr(), y.data_ptr() if want_y else None, q.data_ptr(), rows, H,
                                        gamma.data_ptr(), beta.data_ptr(), 1e-6, fmt, sc.data_ptr(), am.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0
    return y, q, am


@pytest.mark.parametrize("rows,H,limit", [(300, 8192, 1), (64, 16384, 2), (20, 32768, 4), (50, 12288, 2)])
def test_layernorm_single_cta_fallback(dev, hooks_lib, rows, H, limit):
    """With clusters above `limit` counted as not fitting, rows longer than 4096 take the
    single-CTA kernel (gamma and beta read per row): the same bar, from the same call.
    The hook build's give-up index only concerns batch 1 of each CTA, so these shapes
    keep every CTA (and cluster) at one batch."""
    hooks_lib.fp8q_test_set_ln_max_cluster(limit)
    try:
        x = W.residual_stream(seed=H + rows, device=dev, shape=(rows, H))
        gamma, beta = W.layernorm_params(H, seed=H, device=dev)
        y, q, am = _hooked_layernorm(hooks_lib, x, gamma, beta, E4M3FN, 0.017, dev, True)
    finally:
        hooks_lib.fp8q_test_set_ln_max_cluster(0)
    assert cluster_size(H) > limit
    yb = W.bf16_bits(y)
    assert_layernorm_y(W.bf16_bits(x), H, gamma.cpu().numpy(), beta.cpu().numpy(), 1e-6, yb, f"fallback {rows}x{H}")
    rq, ra = par_quantize_amax(yb, E4M3FN, np.float32(0.017))
    assert_codes_equal(q.cpu().numpy(), rq, E4M3FN, f"fallback q {rows}x{H}")
    assert_f32_equal([float(am)], [ra], f"fallback amax {rows}x{H}")
