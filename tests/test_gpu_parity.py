"""GPU parity: libfp8q (through its C ABI) against the CPU oracle.

Bar: bit-exact FP8 codes, amax, history, scale, scale_inv and bf16 dequant.
Where several encodings are equally correct (a NaN), both sides must agree
that the value is a NaN.  Every case compares every element, the full-size
workloads included (the oracle runs chunked over all host cores there).
The producers fused with the quantize are tested in test_gpu_producers.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (CANARY, GUARD, SCALES_ALL, assert_bf16_equal, assert_codes_equal,  # noqa: F401
                         assert_f32_equal, check_guards, check_quantize_full, f32, guarded, is_nan_code,
                         oracle_scale_from, par_dequantize, par_qdq_amax, par_quantize_amax)
from quantize_amax_scaling_gb300 import fp8q
from quantize_amax_scaling_gb300 import workloads as W

pytestmark = pytest.mark.gpu

E4M3FN, E5M2 = fp8q.E4M3FN, fp8q.E5M2


@pytest.fixture(scope="module")
def dev():
    fp8q.lib()
    return torch.device("cuda:0")


def run_quantize(x, fmt, scale, dev, q=None, amax0=0.0):
    if q is None:
        q = torch.empty(x.numel(), dtype=torch.uint8, device=dev)
    am = f32(amax0, dev)
    fp8q.fp8q_quantize_amax(x.reshape(-1), q, fmt, f32(scale, dev), am)
    torch.cuda.synchronize()
    return q, am


# --------------------------------------------------------------------------- quantize

@pytest.mark.parametrize("fmt", [E4M3FN, E5M2])
def test_quantize_every_bf16_pattern_many_scales(dev, fmt):
    x = W.all_bf16_patterns(dev)
    xb = W.bf16_bits(x)
    for s in SCALES_ALL:
        q, am = run_quantize(x, fmt, s, dev)
        rq, ra = oracle.quantize_amax(xb, fmt, np.float32(s))
        assert_codes_equal(q.cpu().numpy(), rq, fmt, f"scale {s!r}")
        assert math.isnan(float(am)) and math.isnan(float(ra))


def test_amax_exact_on_pattern_subsets(dev):
    allx = W.bf16_bits(W.all_bf16_patterns())
    f = (allx.astype(np.uint32) << 16).view(np.float32)
    subsets = {
        "finite": allx[np.isfinite(f)],
        "with_inf": allx[~np.isnan(f)],
        "subnormal": allx[(np.abs(f) < 2.0 ** -126)],
        "negative_only": allx[np.isfinite(f) & (f < 0)],
        "zeros": np.array([0x8000, 0x0000, 0x8000], np.uint16),
    }
    for name, bits in subsets.items():
        x = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(dev)
        q, am = run_quantize(x, E4M3FN, 1.0, dev)
        rq, ra = oracle.quantize_amax(bits, E4M3FN, 1.0)
        assert_f32_equal([float(am)], [ra], name)
        assert_codes_equal(q.cpu().numpy(), rq, E4M3FN, name)


def test_amax_accumulates_into_seed(dev):
    x = W.mlp_activation(7, dev, (64, 256))
    xb = W.bf16_bits(x)
    for seed in (0.0, 0.5, 1e6, math.inf):
        _, am = run_quantize(x, E4M3FN, 1.0, dev, amax0=seed)
        _, ra = oracle.quantize_amax(xb, E4M3FN, 1.0, amax=seed)
        assert_f32_equal([float(am)], [ra], f"seed {seed}")


SIZES = [1, 2, 7, 8, 9, 15, 16, 17, 31, 32, 33, 255, 4095, 4097, 8191, 8192, 8193, 2 * 65536 + 5,
         (1 << 20) + 3]
OFFSETS = [(0, 0), (1, 1), (3, 3), (7, 7), (0, 1), (1, 0), (5, 2), (2, 13), (4, 4), (6, 14),
           (8, 8), (15, 15), (9, 1), (12, 12), (8, 0)]


@pytest.mark.parametrize("n", SIZES)
def test_quantize_ragged_sizes_offsets_with_canaries(dev, n):
    g = torch.Generator(device=dev)
    g.manual_seed(n)
    for k, (xo, qo) in enumerate(OFFSETS if n < 100000 else OFFSETS[:4]):
        fmt = E4M3FN if k % 2 == 0 else E5M2
        scale = [0.0123, 1.0, 2.0 ** 70, 3.3e-3][k % 4]   # includes a slow-path scale
        xbuf = torch.randn(n + 16, generator=g, device=dev).mul_(40.0).to(torch.bfloat16)
        x = xbuf[xo: xo + n]
        qbuf, q = guarded(n, torch.uint8, dev, qo)
        am = f32(0.0, dev)
        fp8q.fp8q_quantize_amax(x, q, fmt, f32(scale, dev), am)
        torch.cuda.synchronize()
        rq, ra = oracle.quantize_amax(W.bf16_bits(x), fmt, np.float32(scale))
        assert_codes_equal(q.cpu().numpy(), rq, fmt, f"n={n} off={xo},{qo}")
        assert_f32_equal([float(am)], [ra], f"amax n={n} off={xo},{qo}")
        check_guards(qbuf, n, qo)


@pytest.mark.parametrize("n,xo,qo", [(16384 + 17, 0, 0), (3 * 16384 + 5, 3, 3), ((1 << 25) + 7, 1, 1),
                                     (2560 * 16384, 0, 0), (2560 * 16384 + 16, 0, 0), (2560 * 16384 + 16, 5, 5),
                                     (2560 * 16384 - 1, 7, 7)])
def test_quantize_both_grids_around_the_threshold(dev, n, xo, qo):
    """Single tensors of up to 2560 tiles take the persistent grid-stride grid,
    larger ones one CTA per tile: both sides of the switch, with heads and tails."""
    g = torch.Generator(device=dev)
    g.manual_seed(n % 100003)
    xbuf = (torch.randn(n + 16, generator=g, device=dev) * 7.0).to(torch.bfloat16)
    x = xbuf[xo: xo + n]
    qbuf, q = guarded(n, torch.uint8, dev, qo)
    for fmt, scale in ((E4M3FN, 0.0123), (E5M2, 2.0 ** 70)):
        am = f32(0.0, dev)
        fp8q.fp8q_quantize_amax(x, q, fmt, f32(scale, dev), am)
        torch.cuda.synchronize()
        check_quantize_full(x, q, am, fmt, np.float32(scale), f"n={n} off={xo},{qo}")
        check_guards(qbuf, n, qo)


def test_quantize_on_a_side_stream(dev):
    x = W.mlp_activation(3, dev, (512, 1024))
    s = torch.cuda.Stream()
    q = torch.empty(x.numel(), dtype=torch.uint8, device=dev)
    am = f32(0.0, dev)
    sc = f32(0.05, dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        fp8q.fp8q_quantize_amax(x.reshape(-1), q, E4M3FN, sc, am, stream=s)
    s.synchronize()
    rq, ra = oracle.quantize_amax(W.bf16_bits(x), E4M3FN, np.float32(0.05))
    assert_codes_equal(q.cpu().numpy(), rq, E4M3FN)
    assert float(am) == float(ra)


def test_tiny_config_page_example(dev):
    """bf16 A 16x32 and B 32x64 from U[0,1), e4m3fn with scale 1, amax per tensor,
    then one scale update (history 16 of zeros, margin 0, max)."""
    A, B = W.tiny_pair(dev)
    amax = torch.zeros(2, device=dev)
    for i, X in enumerate((A, B)):
        q = torch.empty(X.numel(), dtype=torch.uint8, device=dev)
        fp8q.fp8q_quantize_amax(X.reshape(-1), q, E4M3FN, f32(1.0, dev), amax[i:i + 1])
        torch.cuda.synchronize()
        rq, ra = oracle.quantize_amax(W.bf16_bits(X), E4M3FN, 1.0)
        assert_codes_equal(q.cpu().numpy(), rq, E4M3FN)
        assert float(amax[i]) == float(ra)
    hist = torch.zeros(16, 2, device=dev)
    sc = torch.ones(2, device=dev)
    si = torch.ones(2, device=dev)
    fp8q.fp8q_amax_scale_update(hist, amax, sc, si, E4M3FN, fp8q.ALGO_MAX, 0)
    torch.cuda.synchronize()
    rh = np.zeros((16, 2), np.float32)
    rs, ri = np.ones(2, np.float32), np.ones(2, np.float32)
    oracle.amax_scale_update(rh, amax.cpu().numpy(), rs, ri)
    assert_f32_equal(hist.cpu().numpy(), rh, "history")
    assert_f32_equal(sc.cpu().numpy(), rs, "scale")
    assert_f32_equal(si.cpu().numpy(), ri, "scale_inv")


def test_mlp_activation_full_size_full_compare(dev):
    """8192x4096 N(0,1) with 0.1% outliers x100, e4m3fn, delayed scale from the
    previous step's amax -- every byte compared."""
    prev = W.mlp_activation(W.SEED_MLP + 1, dev)
    scale = oracle_scale_from(oracle.amax(W.bf16_bits(prev)), E4M3FN)
    x = W.mlp_activation(W.SEED_MLP, dev)
    q, am = run_quantize(x, E4M3FN, scale, dev)
    xb = W.bf16_bits(x)
    rq, ra = oracle.quantize_amax(xb, E4M3FN, scale)
    assert_codes_equal(q.cpu().numpy(), rq, E4M3FN, "mlp activation")
    assert float(am) == float(ra)


def test_ffn_full_size_multi_tensor(dev):
    """gelu activation 8192x16384 + W1 4096x16384 + W2 16384x4096 in one launch,
    each with its own delayed scale and amax: every code compared."""
    xs = W.ffn_tensors(dev)
    prev = W.ffn_tensors(dev, seed=W.SEED_FFN + 1)
    scales = [oracle_scale_from(oracle.amax(W.bf16_bits(p)), E4M3FN) for p in prev]
    del prev
    qs = [torch.empty(x.numel(), dtype=torch.uint8, device=dev) for x in xs]
    am = torch.zeros(len(xs), device=dev)
    sc = torch.tensor(scales, dtype=torch.float32, device=dev)
    fp8q.fp8q_multi_quantize_amax([x.reshape(-1) for x in xs], qs, E4M3FN,
                                  [sc[i:i + 1] for i in range(3)], [am[i:i + 1] for i in range(3)])
    torch.cuda.synchronize()
    for i, (x, q) in enumerate(zip(xs, qs)):
        check_quantize_full(x, q, am[i], E4M3FN, scales[i], f"ffn tensor {i}")


def test_headline_tensor_single_call(dev):
    """The 8192x16384 activation through the single-tensor entry point: every code."""
    x = W.gelu_activation(W.SEED_FFN, dev)
    scale = np.float32(0.0091)
    q, am = run_quantize(x, E4M3FN, scale, dev)
    check_quantize_full(x, q, am, E4M3FN, scale, "8192x16384")


def test_gradients_e5m2_quantize_then_dequantize(dev):
    """sign x lognormal(-12, 3) gradients with signed zeros and +-inf, e5m2
    saturating (amax = inf), then dequantized back to bf16: every element."""
    grads = W.gradient_tensors(dev)
    prev = W.gradient_tensors(dev, seed=W.SEED_GRAD + 1)
    for g, p in zip(grads, prev):
        pb = W.bf16_bits(p)
        pf = (pb.astype(np.uint32) << 16).view(np.float32)
        finite_prev = pb[np.isfinite(pf)]
        scale = oracle_scale_from(oracle.amax(finite_prev), E5M2)
        q, am = run_quantize(g, E5M2, scale, dev)
        assert math.isinf(float(am))
        rq = check_quantize_full(g, q, am, E5M2, scale, "gradient")
        y = torch.empty(g.numel(), dtype=torch.bfloat16, device=dev)
        fp8q.fp8q_dequantize(q, y, E5M2, f32(scale, dev))
        torch.cuda.synchronize()
        assert_bf16_equal(W.bf16_bits(y), par_dequantize(rq, E5M2, scale), "gradient dequant")


# --------------------------------------------------------------------------- multi-tensor

def _multi_case(dev, sizes, fmt, seed, offsets=True, share_amax=False):
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    rng = np.random.default_rng(seed)
    xs, qs, qbufs, qoffs, scales = [], [], [], [], []
    for i, n in enumerate(sizes):
        xo = int(rng.integers(0, 8)) if offsets else 0
        qo = int(rng.integers(0, 16)) if offsets else 0
        xbuf = (torch.randn(n + 8, generator=g, device=dev) * float(rng.uniform(0.1, 500))).to(torch.bfloat16)
        xs.append(xbuf[xo: xo + n])
        qb, q = guarded(n, torch.uint8, dev, qo)
        qs.append(q)
        qbufs.append(qb)
        qoffs.append(qo)
        scales.append(np.float32([0.01, 1.0, 0.37, 2.0 ** -65, 3.0][i % 5]))
    T = len(sizes)
    sc = torch.tensor(scales, dtype=torch.float32, device=dev)
    am = torch.zeros(T, device=dev)
    amax_views = [am[0:1] if share_amax else am[i:i + 1] for i in range(T)]
    fp8q.fp8q_multi_quantize_amax(xs, qs, fmt, [sc[i:i + 1] for i in range(T)], amax_views)
    torch.cuda.synchronize()
    rqs, ras = oracle.multi_quantize_amax([W.bf16_bits(x) for x in xs], fmt, scales)
    for i in range(T):
        assert_codes_equal(qs[i].cpu().numpy(), rqs[i], fmt, f"tensor {i} of {T}")
        check_guards(qbufs[i], sizes[i], qoffs[i])
    amh = am.cpu().numpy()
    if share_amax:
        want = max((float(a) for a in ras if not math.isnan(a)), default=0.0)
        assert amh[0] == np.float32(want)
    else:
        assert_f32_equal(amh, ras, "amax")


@pytest.mark.parametrize("count", [1, 2, 8, 9, 64, 65, 200, 512])
def test_multi_tensor_every_bucket(dev, count):
    rng = np.random.default_rng(count)
    sizes = [int(v) for v in rng.integers(0, 3000, count)]
    sizes[0] = max(sizes[0], 1)
    _multi_case(dev, sizes, E4M3FN if count % 2 else E5M2, seed=count)


def test_multi_tensor_mixed_large_and_tiny_with_empty(dev):
    sizes = [0, 1, 70000, 3, 0, 8192 * 5 + 7, 9, 123457, 0, 16]
    _multi_case(dev, sizes, E4M3FN, seed=42)
    _multi_case(dev, sizes, E5M2, seed=43, offsets=False)


def test_multi_tensor_shared_amax(dev):
    _multi_case(dev, [5000, 7000, 11, 90000], E4M3FN, seed=44, share_amax=True)


def test_ragged_twelve_tensors_full_size(dev):
    """Twelve bf16 N(0,1) tensors 2048x12288 .. 12288x4096 in one launch, with
    the per-slot scales that a 576-slot update produces: every code."""
    xs = W.ragged_tensors(dev)
    hist, new, sc0, si0, sf = W.scale_update_inputs("cpu")
    hist_np, new_np = hist.numpy().copy(), new.numpy().copy()
    s_np, si_np = sc0.numpy().copy(), si0.numpy().copy()
    oracle.amax_scale_update(hist_np, new_np, s_np, si_np, E4M3FN, oracle.ALGO_MAX, 0)
    scales = [np.float32(s_np[i]) for i in range(len(xs))]
    qs = [torch.empty(x.numel(), dtype=torch.uint8, device=dev) for x in xs]
    am = torch.zeros(len(xs), device=dev)
    sc = torch.tensor(scales, dtype=torch.float32, device=dev)
    fp8q.fp8q_multi_quantize_amax([x.reshape(-1) for x in xs], qs, E4M3FN,
                                  [sc[i:i + 1] for i in range(len(xs))],
                                  [am[i:i + 1] for i in range(len(xs))])
    torch.cuda.synchronize()
    for i, (x, q) in enumerate(zip(xs, qs)):
        check_quantize_full(x, q, am[i], E4M3FN, scales[i], f"ragged {i}")


# --------------------------------------------------------------------------- dequantize

@pytest.mark.parametrize("fmt", [E4M3FN, E5M2])
def test_dequantize_every_code_many_scales(dev, fmt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).repeat(37).to(dev)
    for s in SCALES_ALL:
        y = torch.empty(codes.numel(), dtype=torch.bfloat16, device=dev)
        fp8q.fp8q_dequantize(codes, y, fmt, f32(s, dev))
        torch.cuda.synchronize()
        ry = oracle.dequantize(codes.cpu().numpy(), fmt, np.float32(s))
        assert_bf16_equal(W.bf16_bits(y), ry, f"scale {s!r}")


@pytest.mark.parametrize("n", SIZES)
def test_dequantize_ragged_sizes_offsets_with_canaries(dev, n):
    rng = np.random.default_rng(n)
    for k, (qo, yo) in enumerate(OFFSETS if n < 100000 else OFFSETS[:4]):
        fmt = E4M3FN if k % 2 == 0 else E5M2
        qbuf = torch.from_numpy(rng.integers(0, 256, n + 16, dtype=np.uint8)).to(dev)
        q = qbuf[qo: qo + n]
        ybuf, y = guarded(n, torch.bfloat16, dev, yo, fill=0x5A5A)
        s = [0.0123, 1.0, 3.0e5, 2.0 ** -100][k % 4]
        fp8q.fp8q_dequantize(q, y, fmt, f32(s, dev))
        torch.cuda.synchronize()
        ry = oracle.dequantize(q.cpu().numpy(), fmt, np.float32(s))
        assert_bf16_equal(W.bf16_bits(y), ry, f"n={n} off={qo},{yo}")
        check_guards(ybuf, n, yo, fill=0x5A5A)


# --------------------------------------------------------------------------- scale update

def _update_case(dev, hist_np, new_np, fmt=E4M3FN, algo=0, margin=0, slot_format=None, steps=1,
                 scale0=None, hist_offset=0):
    H, S = hist_np.shape
    if hist_offset:
        buf = torch.zeros(H * S + hist_offset, device=dev)
        hist = buf[hist_offset:].view(H, S)
        hist.copy_(torch.from_numpy(hist_np))
    else:
        hist = torch.from_numpy(hist_np.copy()).to(dev)
    sc = torch.from_numpy(scale0.copy() if scale0 is not None else np.ones(S, np.float32)).to(dev)
    si = torch.from_numpy((1.0 / sc.cpu().numpy()).astype(np.float32)).to(dev)
    rh = hist_np.copy()
    rs, ri = sc.cpu().numpy().copy(), si.cpu().numpy().copy()
    sf_t = None if slot_format is None else torch.from_numpy(slot_format).to(dev)
    for step in range(steps):
        with np.errstate(over="ignore"):  # large specials overflow to inf on purpose
            new_s = new_np if step == 0 else np.roll(new_np, step) * np.float32(1.5 ** step)
        new_t = torch.from_numpy(np.ascontiguousarray(new_s, np.float32)).to(dev)
        fp8q.fp8q_amax_scale_update(hist, new_t, sc, si, fmt, algo, margin, sf_t)
        oracle.amax_scale_update(rh, new_s, rs, ri, fmt, algo, margin, slot_format)
    torch.cuda.synchronize()
    assert_f32_equal(hist.cpu().numpy(), rh, f"history {H}x{S}")
    assert_f32_equal(sc.cpu().numpy(), rs, f"scale {H}x{S}")
    assert_f32_equal(si.cpu().numpy(), ri, f"scale_inv {H}x{S}")


@pytest.mark.parametrize("algo", [fp8q.ALGO_MAX, fp8q.ALGO_MOST_RECENT])
@pytest.mark.parametrize("margin", [0, 1])
@pytest.mark.parametrize("per_slot", [False, True])
def test_scale_update_576_slots_full(dev, algo, margin, per_slot):
    """96 layers x 6 slots, history 1024, lognormal(0,2) with 2% zeros."""
    hist, new, _, _, sf = W.scale_update_inputs("cpu")
    _update_case(dev, hist.numpy(), new.numpy(), algo=algo, margin=margin,
                 slot_format=sf.numpy() if per_slot else None, steps=3)


# H up to 1024 takes the one-chunk path, where each thread holds 4 consecutive rows and the
# last one crosses into the next thread's block (and, every 128 rows, the next warp's);
# longer histories stream in chunks.
SHAPES = [(1, 1), (1, 5), (2, 3), (3, 9), (4, 4), (5, 6), (16, 2), (17, 7), (127, 5), (129, 8),
          (257, 3), (513, 16), (1023, 577), (1024, 575), (1025, 576), (1024, 4), (2053, 12), (3000, 8),
          (4096, 4)]


@pytest.mark.parametrize("H,S", SHAPES)
def test_scale_update_shapes(dev, H, S):
    rng = np.random.default_rng(H * 1000 + S)
    hist = np.exp(rng.normal(0, 2, (H, S))).astype(np.float32)
    hist[rng.random((H, S)) < 0.05] = 0.0
    new = np.exp(rng.normal(0, 2, S)).astype(np.float32)
    for algo in (0, 1):
        _update_case(dev, hist, new, algo=algo, margin=(H % 3) - 1, steps=2)


def test_scale_update_misaligned_history_uses_scalar_path(dev):
    rng = np.random.default_rng(8)
    hist = np.exp(rng.normal(0, 2, (1024, 576))).astype(np.float32)
    new = np.exp(rng.normal(0, 2, 576)).astype(np.float32)
    _update_case(dev, hist, new, hist_offset=1, steps=2)


def test_scale_update_specials(dev):
    S = 12
    hist = np.full((8, S), 2.0, np.float32)
    hist[3, 0] = np.nan          # NaN inside the window: pass-through under max
    hist[7, 1] = np.nan          # NaN in the row that drops out: ignored
    hist[2, 2] = np.inf          # inf in the window
    hist[:, 3] = 0.0             # all zero, new zero
    hist[:, 4] = -5.0            # negative history
    new = np.array([1, 1, 1, 0, 1, np.nan, np.inf, -1, 1e-38, 3e38, 1e-45, 448], np.float32)
    scale0 = np.full(S, 4.0, np.float32)
    sf = np.array([0, 1, 0, 0, 1, 0, 1, 0, 0, 1, 0, 5], np.uint8)
    for algo in (0, 1):
        for margin in (-64, -3, 0, 2, 64):
            _update_case(dev, hist, new, algo=algo, margin=margin, slot_format=sf, scale0=scale0,
                         steps=2)


# --------------------------------------------------------------------------- limits and capture

def test_more_than_2_pow_31_elements(dev):
    """Tile and index arithmetic stays 64-bit: quantize, dequantize, the fused quantize ->
    dequantize and the ragged quantize over 2^31 + 4099 elements."""
    n = (1 << 31) + 4099
    g = torch.Generator(device=dev)
    g.manual_seed(31)
    x = torch.empty(n, dtype=torch.bfloat16, device=dev)
    chunk = 1 << 28
    for i in range(0, n, chunk):          # draw in chunks to bound the float32 temporary
        m = min(chunk, n - i)
        x[i:i + m] = (torch.randn(m, generator=g, device=dev) * 3.0).to(torch.bfloat16)
    x[n - 1] = 1000.0                     # the largest magnitude sits in the last element
    q = torch.empty(n, dtype=torch.uint8, device=dev)
    scale = np.float32(0.37)
    am = f32(0.0, dev)
    fp8q.fp8q_quantize_amax(x, q, E4M3FN, f32(scale, dev), am)
    y = torch.empty(n, dtype=torch.bfloat16, device=dev)
    fp8q.fp8q_dequantize(q, y, E4M3FN, f32(scale, dev))
    torch.cuda.synchronize()
    assert float(am) == 1000.0
    chunk = 1 << 28
    for i in range(0, n, chunk):          # every element, a host chunk at a time
        m = min(chunk, n - i)
        rq, _ = par_quantize_amax(W.bf16_bits(x[i:i + m]), E4M3FN, scale)
        assert_codes_equal(q[i:i + m].cpu().numpy(), rq, E4M3FN, f"n > 2^31, chunk at {i}")
        assert_bf16_equal(W.bf16_bits(y[i:i + m]), par_dequantize(rq, E4M3FN, scale), f"dequant chunk at {i}")
    # the fused quantize -> dequantize equals the two calls, and the ragged path over a list of
    # a small tensor and this one equals the single calls
    y2 = torch.empty(n, dtype=torch.bfloat16, device=dev)
    am2 = f32(0.0, dev)
    fp8q.fp8q_qdq_amax(x, y2, E4M3FN, f32(scale, dev), am2)
    small = x[: 3 * 16384 + 5].clone()
    qs, q2 = torch.empty_like(small, dtype=torch.uint8), torch.empty_like(q)
    ams = torch.zeros(2, device=dev)
    fp8q.fp8q_multi_quantize_amax([small, x], [qs, q2], E4M3FN, [f32(scale, dev), f32(scale, dev)],
                                  [ams[0:1], ams[1:2]])
    torch.cuda.synchronize()
    assert torch.equal(y2.view(torch.int16), y.view(torch.int16)) and float(am2) == 1000.0
    assert torch.equal(q2, q) and float(ams[1]) == 1000.0
    assert torch.equal(qs, q[: small.numel()])
    del x, q, y, y2, q2
    torch.cuda.empty_cache()


def test_step_captured_in_a_cuda_graph(dev):
    """Quantize, ragged quantize, dequantize and the update, captured once and replayed:
    the calls enqueue device work only, so a graph replays them bit-exactly."""
    act = W.mlp_activation(11, dev, (256, 1024)).reshape(-1)
    ws = [W.truncated_normal_weight((64, 1024), 1024, 12, dev).reshape(-1),
          W.truncated_normal_weight((1024, 33), 1024, 13, dev).reshape(-1)]
    grad_q = torch.from_numpy(np.random.default_rng(3).integers(0, 256, 5000, dtype=np.uint8)).to(dev)
    H, S = 16, 8
    hist = torch.zeros(H, S, device=dev)
    amax = torch.zeros(S, device=dev)
    scale = torch.ones(S, device=dev)
    scale_inv = torch.ones(S, device=dev)
    q_act = torch.empty(act.numel(), dtype=torch.uint8, device=dev)
    q_w = [torch.empty(w.numel(), dtype=torch.uint8, device=dev) for w in ws]
    y = torch.empty(grad_q.numel(), dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream()

    def step():
        amax[:3].zero_()
        fp8q.fp8q_quantize_amax(act, q_act, E4M3FN, scale[0:1], amax[0:1], stream=s)
        fp8q.fp8q_multi_quantize_amax(ws, q_w, E4M3FN, [scale[1:2], scale[2:3]], [amax[1:2], amax[2:3]],
                                      stream=s)
        fp8q.fp8q_dequantize(grad_q, y, E5M2, scale[3:4], stream=s)
        fp8q.fp8q_amax_scale_update(hist, amax, scale, scale_inv, E4M3FN, fp8q.ALGO_MAX, 0, stream=s)

    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        step()                      # first call on this device (caches launch geometry)
    s.synchronize()
    hist.zero_(); amax.zero_(); scale.fill_(1.0); scale_inv.fill_(1.0)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    # oracle: three steps of delayed scaling
    rh = np.zeros((H, S), np.float32)
    ra = np.zeros(S, np.float32)
    rs, ri = np.ones(S, np.float32), np.ones(S, np.float32)
    xa, xw = W.bf16_bits(act), [W.bf16_bits(w) for w in ws]
    gq = grad_q.cpu().numpy()
    for _ in range(3):
        graph.replay()
        torch.cuda.synchronize()
        sc = rs.copy()
        rq_act, a0 = oracle.quantize_amax(xa, E4M3FN, sc[0])
        rq_w, aw = oracle.multi_quantize_amax(xw, E4M3FN, [sc[1], sc[2]])
        ry = oracle.dequantize(gq, E5M2, sc[3])
        ra[:3] = [a0, aw[0], aw[1]]
        oracle.amax_scale_update(rh, ra, rs, ri, E4M3FN, oracle.ALGO_MAX, 0)
        assert_codes_equal(q_act.cpu().numpy(), rq_act, E4M3FN, "graph act")
        for qq, rr in zip(q_w, rq_w):
            assert_codes_equal(qq.cpu().numpy(), rr, E4M3FN, "graph weights")
        assert_bf16_equal(W.bf16_bits(y), ry, "graph dequant")
        assert_f32_equal(hist.cpu().numpy(), rh, "graph history")
        assert_f32_equal(scale.cpu().numpy(), rs, "graph scale")
        assert_f32_equal(scale_inv.cpu().numpy(), ri, "graph scale_inv")


# --------------------------------------------------------------------------- fused Q -> DQ

def run_qdq(x, fmt, scale, dev, y=None, amax0=0.0):
    if y is None:
        y = torch.empty(x.numel(), dtype=torch.bfloat16, device=dev)
    am = f32(amax0, dev)
    fp8q.fp8q_qdq_amax(x.reshape(-1), y, fmt, f32(scale, dev), am)
    torch.cuda.synchronize()
    return y, am


@pytest.mark.parametrize("fmt", [E4M3FN, E5M2])
def test_qdq_every_bf16_pattern_many_scales(dev, fmt):
    x = W.all_bf16_patterns(dev)
    xb = W.bf16_bits(x)
    for s in SCALES_ALL:
        y, am = run_qdq(x, fmt, s, dev)
        ry, ra = oracle.qdq_amax(xb, fmt, np.float32(s))
        assert_bf16_equal(W.bf16_bits(y), ry, f"scale {s!r}")
        assert math.isnan(float(am)) and math.isnan(float(ra))


@pytest.mark.parametrize("n", [1, 15, 16, 17, 33, 4095, 8193, (1 << 20) + 3])
def test_qdq_sizes_offsets_in_place_and_canaries(dev, n):
    g = torch.Generator(device=dev)
    g.manual_seed(7 * n)
    for k, (xo, yo) in enumerate(OFFSETS if n < 100000 else OFFSETS[:4]):
        fmt = E4M3FN if k % 2 else E5M2
        scale = [0.0123, 1.0, 2.0 ** 70, 3.3e-3][k % 4]
        xbuf = (torch.randn(n + 16, generator=g, device=dev) * 30.0).to(torch.bfloat16)
        x = xbuf[xo: xo + n]
        ybuf, y = guarded(n, torch.bfloat16, dev, yo, fill=0x5A5A)
        am = f32(0.0, dev)
        fp8q.fp8q_qdq_amax(x, y, fmt, f32(scale, dev), am)
        torch.cuda.synchronize()
        xb = W.bf16_bits(x)
        ry, ra = oracle.qdq_amax(xb, fmt, np.float32(scale))
        assert_bf16_equal(W.bf16_bits(y), ry, f"n={n} off={xo},{yo}")
        assert_f32_equal([float(am)], [ra], f"amax n={n}")
        check_guards(ybuf, n, yo, fill=0x5A5A)
        # in place: y is x
        am2 = f32(0.0, dev)
        fp8q.fp8q_qdq_amax(x, x, fmt, f32(scale, dev), am2)
        torch.cuda.synchronize()
        assert_bf16_equal(W.bf16_bits(x), ry, f"in place n={n}")
        assert_f32_equal([float(am2)], [ra], f"in-place amax n={n}")


def test_qdq_full_size_activation(dev):
    x = W.gelu_activation(W.SEED_FFN, dev).reshape(-1)
    scale = np.float32(0.0091)
    y, am = run_qdq(x, E4M3FN, scale, dev)
    ry, ra = par_qdq_amax(W.bf16_bits(x), E4M3FN, scale)
    assert_bf16_equal(W.bf16_bits(y), ry, "qdq 8192x16384")
    assert_f32_equal([float(am)], [ra], "qdq amax")


# --------------------------------------------------------------------------- ring-buffer history

def _ring_case(dev, hist_np, head_np, new_np, algo=0, margin=0, slot_format=None, steps=1,
               scale0=None, hist_offset=0):
    H, S = hist_np.shape
    if hist_offset:
        buf = torch.zeros(H * S + hist_offset, device=dev)
        hist = buf[hist_offset:].view(H, S)
        hist.copy_(torch.from_numpy(hist_np))
    else:
        hist = torch.from_numpy(hist_np.copy()).to(dev)
    head = torch.from_numpy(head_np.copy()).to(dev)
    s0 = scale0 if scale0 is not None else np.ones(S, np.float32)
    sc = torch.from_numpy(s0.copy()).to(dev)
    si = torch.from_numpy((1.0 / s0).astype(np.float32)).to(dev)
    rh, rhead = hist_np.copy(), head_np.copy()
    rs, ri = sc.cpu().numpy().copy(), si.cpu().numpy().copy()
    sf_t = None if slot_format is None else torch.from_numpy(slot_format).to(dev)
    for step in range(steps):
        with np.errstate(over="ignore"):  # large specials overflow to inf on purpose
            new_s = new_np if step == 0 else (np.roll(new_np, step) * np.float32(1.25 ** step)).astype(np.float32)
        fp8q.fp8q_amax_scale_update_ring(hist, head, torch.from_numpy(new_s).to(dev), sc, si, E4M3FN, algo,
                                         margin, sf_t)
        oracle.amax_scale_update_ring(rh, rhead, new_s, rs, ri, E4M3FN, algo, margin, slot_format)
    torch.cuda.synchronize()
    assert np.array_equal(head.cpu().numpy(), rhead), "head"
    assert_f32_equal(hist.cpu().numpy(), rh, f"ring history {H}x{S}")
    assert_f32_equal(sc.cpu().numpy(), rs, f"ring scale {H}x{S}")
    assert_f32_equal(si.cpu().numpy(), ri, f"ring scale_inv {H}x{S}")


@pytest.mark.parametrize("algo", [fp8q.ALGO_MAX, fp8q.ALGO_MOST_RECENT])
@pytest.mark.parametrize("margin", [0, 1])
@pytest.mark.parametrize("per_slot", [False, True])
def test_ring_update_576_slots_full(dev, algo, margin, per_slot):
    hist, new, _, _, sf = W.scale_update_inputs("cpu")
    H, S = hist.shape
    head = np.random.default_rng(5).integers(0, H, S).astype(np.int32)
    _ring_case(dev, hist.numpy(), head, new.numpy(), algo=algo, margin=margin,
               slot_format=sf.numpy() if per_slot else None, steps=3)


@pytest.mark.parametrize("H,S", SHAPES)
def test_ring_update_shapes(dev, H, S):
    rng = np.random.default_rng(H * 7 + S)
    hist = np.exp(rng.normal(0, 2, (H, S))).astype(np.float32)
    hist[rng.random((H, S)) < 0.05] = 0.0
    new = np.exp(rng.normal(0, 2, S)).astype(np.float32)
    head = rng.integers(0, H, S).astype(np.int32)
    for algo in (0, 1):
        _ring_case(dev, hist, head, new, algo=algo, margin=(H % 3) - 1, steps=2)


def test_ring_update_specials_corrupt_heads_and_scalar_path(dev):
    S = 12
    hist = np.full((8, S), 2.0, np.float32)
    hist[3, 0] = np.nan
    hist[2, 2] = np.inf
    hist[:, 3] = 0.0
    new = np.array([1, 1, 1, 0, 1, np.nan, np.inf, -1, 1e-38, 3e38, 1e-45, 448], np.float32)
    head = np.array([7, 3, 0, 5, -1, 8, 2, 2, 2, 2, 2, 1000], np.int32)   # -1, 8, 1000 are corrupt
    sf = np.array([0, 1, 0, 0, 1, 0, 1, 0, 0, 1, 0, 5], np.uint8)
    for algo in (0, 1):
        _ring_case(dev, hist, head, new, algo=algo, slot_format=sf, scale0=np.full(S, 4.0, np.float32), steps=2)
    rng = np.random.default_rng(9)
    big = np.exp(rng.normal(0, 2, (1024, 576))).astype(np.float32)
    _ring_case(dev, big, rng.integers(0, 1024, 576).astype(np.int32),
               np.exp(rng.normal(0, 2, 576)).astype(np.float32), hist_offset=1, steps=2)


def test_ring_matches_roll_on_the_gpu(dev):
    """Both GPU forms, fed the same amaxes, give the same window (unrotated) and scales."""
    hist, new, _, _, sf = W.scale_update_inputs(dev)
    H, S = hist.shape
    roll = hist.clone()
    ring = hist.flip(0).contiguous()             # newest row at the bottom ...
    head = torch.full((S,), H - 1, dtype=torch.int32, device=dev)   # ... where head points
    sc_a, si_a = torch.ones(S, device=dev), torch.ones(S, device=dev)
    sc_b, si_b = sc_a.clone(), si_a.clone()
    g = torch.Generator(device=dev)
    g.manual_seed(77)
    for _ in range(5):
        a = torch.exp(torch.randn(S, generator=g, device=dev) * 2)
        fp8q.fp8q_amax_scale_update(roll, a, sc_a, si_a, E4M3FN, fp8q.ALGO_MAX, 0, sf)
        fp8q.fp8q_amax_scale_update_ring(ring, head, a, sc_b, si_b, E4M3FN, fp8q.ALGO_MAX, 0, sf)
    torch.cuda.synchronize()
    h = head.cpu().numpy()
    rg = ring.cpu().numpy()
    logical = np.stack([rg[(h - r) % H, np.arange(S)] for r in range(H)])
    assert_f32_equal(logical, roll.cpu().numpy(), "ring vs roll window")
    assert_f32_equal(sc_b.cpu().numpy(), sc_a.cpu().numpy(), "ring vs roll scale")
    assert_f32_equal(si_b.cpu().numpy(), si_a.cpu().numpy(), "ring vs roll scale_inv")


# --------------------------------------------------------------------------- update fused with the next quantize

def _fused_case(dev, H, S, slot, n, algo=0, margin=0, per_slot=False, steps=2, seed=0, specials=None,
                scale0=None):
    """Run fp8q_amax_scale_update_ring_quantize `steps` times (heads swapped between
    calls, a new x each step) beside the oracle's update-then-quantize."""
    rng = np.random.default_rng(seed)
    hist_np = np.exp(rng.normal(0, 2, (H, S))).astype(np.float32)
    hist_np[rng.random((H, S)) < 0.02] = 0.0
    head_np = rng.integers(0, H, S).astype(np.int32)
    sf_np = (np.arange(S) % 6 >= 4).astype(np.uint8) if per_slot else None
    fmt = int(sf_np[slot]) if per_slot else E4M3FN
    s0 = scale0 if scale0 is not None else np.exp(rng.normal(0, 1, S)).astype(np.float32)
    hist = torch.from_numpy(hist_np.copy()).to(dev)
    heads = [torch.from_numpy(head_np.copy()).to(dev), torch.full((S,), -7, dtype=torch.int32, device=dev)]
    sc = torch.from_numpy(s0.copy()).to(dev)
    si = torch.from_numpy((1.0 / s0).astype(np.float32)).to(dev)
    sf = None if sf_np is None else torch.from_numpy(sf_np).to(dev)
    rh, rhead, rs, ri = hist_np.copy(), head_np.copy(), s0.copy(), (1.0 / s0).astype(np.float32)
    g = torch.Generator(device=dev)
    for step in range(steps):
        new_np = np.exp(rng.normal(0, 2, S)).astype(np.float32)
        if specials is not None:
            specials(step, new_np, heads[step % 2], rhead)
        g.manual_seed(seed * 100 + step)
        x = (torch.randn(n, generator=g, device=dev) * 3.0).to(torch.bfloat16)
        q = torch.empty(n, dtype=torch.uint8, device=dev)
        am = f32(0.0, dev)
        head_in, head_out = heads[step % 2], heads[(step + 1) % 2]
        before_in = head_in.cpu().numpy().copy()
        fp8q.fp8q_amax_scale_update_ring_quantize(hist, head_in, head_out, torch.from_numpy(new_np).to(dev), sc,
                                                  si, x, q, slot, am, fmt, algo, margin, sf)
        torch.cuda.synchronize()
        rq, ra = oracle.amax_scale_update_ring_quantize(rh, rhead, new_np, rs, ri, W.bf16_bits(x), slot, fmt,
                                                        algo, margin, sf_np)
        what = f"{H}x{S} slot {slot} n {n} algo {algo} margin {margin} step {step}"
        assert np.array_equal(head_in.cpu().numpy(), before_in), "head_in written: " + what
        assert np.array_equal(head_out.cpu().numpy(), rhead), "head_out: " + what
        assert_f32_equal(hist.cpu().numpy(), rh, "history: " + what)
        assert_f32_equal(sc.cpu().numpy(), rs, "scale: " + what)
        assert_f32_equal(si.cpu().numpy(), ri, "scale_inv: " + what)
        assert_codes_equal(q.cpu().numpy(), rq, fmt, "q: " + what)
        assert_f32_equal([float(am)], [ra], "amax: " + what)


@pytest.mark.parametrize("algo", [fp8q.ALGO_MAX, fp8q.ALGO_MOST_RECENT])
@pytest.mark.parametrize("margin", [0, 1])
@pytest.mark.parametrize("per_slot", [False, True])
def test_ring_update_quantize_576_slots(dev, algo, margin, per_slot):
    for k, slot in enumerate((0, 5, 331, 575)):
        _fused_case(dev, 1024, 576, slot, [8193, 2 * 65536 + 5, 1, 1 << 20][k], algo, margin, per_slot,
                    steps=3, seed=11 * k + algo)


@pytest.mark.parametrize("H,S", [(1, 5), (2, 3), (16, 2), (17, 7), (3, 577), (1025, 576)])
def test_ring_update_quantize_shapes(dev, H, S):
    for slot in sorted({0, S // 2, S - 1}):
        _fused_case(dev, H, S, slot, 70001, steps=H + 2 if H < 20 else 2, seed=H * 1000 + S + slot)


def test_ring_update_quantize_empty_tensor_runs_the_update(dev):
    _fused_case(dev, 64, 12, 3, 0, steps=2, seed=5)


def test_ring_update_quantize_pass_through_and_corrupt_heads(dev):
    """The slot's new amax 0, NaN or inf keeps its old scale (the quantize uses it);
    a head outside [0, H) leaves the slot alone and copies its head."""
    S, slot = 10, 4

    def specials(step, new_np, head_in_dev, ref_head):
        if step == 0:
            new_np[slot] = 0.0
        elif step == 1:
            new_np[slot] = np.nan
        elif step == 2:
            new_np[slot] = np.inf
        elif step == 3:
            head_in_dev[slot] = -1
            ref_head[slot] = -1
        elif step == 4:
            head_in_dev[slot] = 32
            ref_head[slot] = 32
    _fused_case(dev, 32, S, slot, 9000, steps=5, seed=3, specials=specials)


def test_ring_update_quantize_equals_the_two_calls(dev):
    """Against the library's own ring update followed by its quantize, on the 96-layer
    history and the full 8192x16384 activation."""
    hist, new, scale, scale_inv, sf = W.scale_update_inputs(dev)
    S = new.numel()
    head = torch.randint(0, hist.shape[0], (S,), dtype=torch.int32, device=dev,
                         generator=torch.Generator(device=dev).manual_seed(1))
    x = W.gelu_activation(W.SEED_FFN, dev).reshape(-1)
    slot = 6 * 40 + 1  # an e4m3fn activation slot
    h1, hd1, s1, i1 = hist.clone(), head.clone(), scale.clone(), scale_inv.clone()
    q1 = torch.empty(x.numel(), dtype=torch.uint8, device=dev)
    a1 = f32(0.0, dev)
    fp8q.fp8q_amax_scale_update_ring(h1, hd1, new, s1, i1, E4M3FN, fp8q.ALGO_MAX, 0, sf)
    fp8q.fp8q_quantize_amax(x, q1, E4M3FN, s1[slot:slot + 1], a1)
    h2, s2, i2 = hist.clone(), scale.clone(), scale_inv.clone()
    hd2 = torch.empty_like(head)
    q2 = torch.empty_like(q1)
    a2 = f32(0.0, dev)
    fp8q.fp8q_amax_scale_update_ring_quantize(h2, head, hd2, new, s2, i2, x, q2, slot, a2, E4M3FN,
                                              fp8q.ALGO_MAX, 0, sf)
    torch.cuda.synchronize()
    assert torch.equal(hd1, hd2) and torch.equal(h1, h2)
    assert torch.equal(s1, s2) and torch.equal(i1, i2)
    assert torch.equal(q1, q2) and float(a1) == float(a2)


def test_fp32_max_grad_example_on_the_gpu(dev):
    """The worked example of the section "Gradient accumulation of FP8 params": x = 2,
    amax history [0, 0, 0], scale 1, three in_qdq iterations accumulating amax with
    max, then one update of the length-3 history."""
    x = torch.full((1,), 2.0, dtype=torch.bfloat16, device=dev)
    y = torch.empty_like(x)
    am = f32(0.0, dev)
    for _ in range(3):
        fp8q.fp8q_qdq_amax(x, y, E4M3FN, f32(1.0, dev), am)
        torch.cuda.synchronize()
        assert float(y) == 2.0
    assert float(am) == 2.0
    hist = torch.zeros(3, 1, device=dev)
    sc, si = torch.ones(1, device=dev), torch.ones(1, device=dev)
    fp8q.fp8q_amax_scale_update(hist, am, sc, si)
    torch.cuda.synchronize()
    assert hist[:, 0].tolist() == [2.0, 0.0, 0.0]
    assert sc.cpu().numpy()[0] == np.float32(2.0) / np.float32(448.0)
