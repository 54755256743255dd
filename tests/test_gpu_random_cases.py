"""Seeded random cases for the streaming calls and the scale updates, every element
against the oracle.

Each case draws its size log-uniformly from 1 element (or from 2^15) to 2^26.5 (so that
every grid form and vector/scalar split comes up: one CTA per tile, the persistent
grid-stride grid, heads and tails), element offsets of input and output from 0 to 15
(mostly equal, so that the vector path runs with a head), the format, a scale
(a third from the special and slow-path scales, the rest 2^U(-40, 40)), an amax seed,
and data of a random magnitude with random special values sprinkled in (signed zeros,
infinities, NaN, bf16 subnormals, the largest finite bf16).  Outputs sit between canary
guards.  The scale updates draw the history's length and slot count, the options, the
amax distribution with specials, the scales and (ring) the heads, corrupt ones included;
the ring update fused with the next quantize draws those, the slot and the tensor's size.
The case parameters come from fixed seeds, so every run draws the same cases.
"""
import math

import numpy as np
import pytest
import torch

from gpu_helpers import (SCALES_ALL, assert_bf16_equal, assert_f32_equal, bf16_bits_of, check_guards,
                         check_quantize_full, combine_amax, f32, guarded, par_dequantize, par_qdq_amax,
                         par_quantize_amax, assert_codes_equal)
from quantize_amax_scaling_gb300 import fp8q
from test_gpu_parity import _fused_case, _ring_case, _update_case

pytestmark = pytest.mark.gpu

E4M3FN, E5M2 = fp8q.E4M3FN, fp8q.E5M2
SPECIAL_BITS = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x0001, 0x8001, 0x007F, 0x7F7F, 0xFF7F],
                        np.uint16)


@pytest.fixture(scope="module")
def dev():
    fp8q.lib()
    return torch.device("cuda:0")


def draw_scale(rng):
    if rng.random() < 1 / 3:
        return float(np.float32(SCALES_ALL[rng.integers(len(SCALES_ALL))]))
    return float(np.float32(2.0 ** rng.uniform(-40, 40)))


def draw_size(rng, top=26.5):
    """log-uniform from 1 element, or (half the time) from 2^15, to 2^top"""
    lo = 15.0 if rng.random() < 0.5 and top > 15 else 0.0
    return max(1, int(2.0 ** rng.uniform(lo, top)))


def draw_offsets(rng):
    """Element offsets of input and output: the same (the vector path, with a head when not
    0) most of the time, else independent (the scalar path when they disagree mod 16)."""
    xo = int(rng.integers(0, 16))
    return xo, (xo if rng.random() < 0.6 else int(rng.integers(0, 16)))


def data_bits(rng, n):
    """bf16 bit patterns: N(0, 1) times 10^U(-4, 4), with up to 64 specials at random places."""
    x = rng.standard_normal(n, dtype=np.float32) * np.float32(10.0 ** rng.uniform(-4, 4))
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    if rng.random() < 0.5:
        k = int(rng.integers(1, 65))
        bits[rng.integers(0, n, k)] = SPECIAL_BITS[rng.integers(0, len(SPECIAL_BITS), k)]
    return bits


def to_device(bits, dev, offset):
    """A bf16 device view of the given bits, starting `offset` elements into its buffer."""
    buf = torch.empty(bits.size + 16, dtype=torch.int16, device=dev)
    view = buf[offset: offset + bits.size]
    view.copy_(torch.from_numpy(bits.view(np.int16)))
    return view.view(torch.bfloat16)


def draw_single(seed):
    rng = np.random.default_rng(seed)
    n = draw_size(rng)
    xo, oo = draw_offsets(rng)
    return dict(n=n, xo=xo, oo=oo,
                fmt=E4M3FN if rng.random() < 0.5 else E5M2, scale=draw_scale(rng),
                amax0=float([0.0, 0.0, 1e-3, 3.0, math.inf][rng.integers(5)]), data_seed=seed * 7 + 1)


QUANTIZE_CASES = [draw_single(1000 + i) for i in range(48)]
QDQ_CASES = [draw_single(2000 + i) for i in range(32)]
DEQUANTIZE_CASES = [draw_single(3000 + i) for i in range(32)]


def case_id(c):
    return f"n{c['n']}-x{c['xo']}-o{c['oo']}-f{c['fmt']}-s{c['scale']:.3g}"


@pytest.mark.parametrize("c", QUANTIZE_CASES, ids=case_id)
def test_random_quantize(dev, c):
    rng = np.random.default_rng(c["data_seed"])
    bits = data_bits(rng, c["n"])
    x = to_device(bits, dev, c["xo"])
    qbuf, q = guarded(c["n"], torch.uint8, dev, c["oo"])
    am = f32(c["amax0"], dev)
    fp8q.fp8q_quantize_amax(x, q, c["fmt"], f32(c["scale"], dev), am)
    torch.cuda.synchronize()
    check_quantize_full(x, q, am, c["fmt"], np.float32(c["scale"]), case_id(c), amax0=c["amax0"])
    check_guards(qbuf, c["n"], c["oo"])


@pytest.mark.parametrize("c", QDQ_CASES, ids=case_id)
def test_random_qdq(dev, c):
    rng = np.random.default_rng(c["data_seed"])
    bits = data_bits(rng, c["n"])
    x = to_device(bits, dev, c["xo"])
    in_place = c["n"] % 3 == 0
    if in_place:
        y = x
    else:
        ybuf, y = guarded(c["n"], torch.bfloat16, dev, c["oo"])
    am = f32(c["amax0"], dev)
    fp8q.fp8q_qdq_amax(x, y, c["fmt"], f32(c["scale"], dev), am)
    torch.cuda.synchronize()
    ry, ra = par_qdq_amax(bits, c["fmt"], np.float32(c["scale"]), c["amax0"])
    assert_bf16_equal(bf16_bits_of(y), ry, case_id(c))
    assert_f32_equal([float(am)], [ra], case_id(c) + " amax")
    if not in_place:
        check_guards(ybuf, c["n"], c["oo"])


@pytest.mark.parametrize("c", DEQUANTIZE_CASES, ids=case_id)
def test_random_dequantize(dev, c):
    rng = np.random.default_rng(c["data_seed"])
    codes = rng.integers(0, 256, c["n"], dtype=np.uint8)
    qbuf = torch.empty(c["n"] + 16, dtype=torch.uint8, device=dev)
    q = qbuf[c["xo"]: c["xo"] + c["n"]]
    q.copy_(torch.from_numpy(codes))
    ybuf, y = guarded(c["n"], torch.bfloat16, dev, c["oo"])
    fp8q.fp8q_dequantize(q, y, c["fmt"], f32(c["scale"], dev))
    torch.cuda.synchronize()
    assert_bf16_equal(bf16_bits_of(y), par_dequantize(codes, c["fmt"], np.float32(c["scale"])), case_id(c))
    check_guards(ybuf, c["n"], c["oo"])


def draw_list(seed):
    rng = np.random.default_rng(seed)
    count = int([1, 2, 3, 12, 40, 64, 65, 300, 512][rng.integers(9)])
    top = 22 if count <= 12 else (18 if count <= 65 else 14)
    sizes = [0 if rng.random() < 0.1 else draw_size(rng, top) for _ in range(count)]
    return dict(count=count, sizes=sizes, fmt=E4M3FN if rng.random() < 0.5 else E5M2,
                **dict(zip(("xo", "oo"), map(list, zip(*[draw_offsets(rng) for _ in range(count)])))),
                scales=[draw_scale(rng) for _ in range(count)],
                shared=rng.random() < 0.3, data_seed=seed * 7 + 3)


LIST_CASES = [draw_list(4000 + i) for i in range(24)]


@pytest.mark.parametrize("c", LIST_CASES, ids=lambda c: f"T{c['count']}-f{c['fmt']}-max{max(c['sizes'])}")
def test_random_multi_tensor_list(dev, c):
    """A ragged list in one launch; with `shared`, every third tensor max-accumulates into
    one amax of the list's first tensor."""
    rng = np.random.default_rng(c["data_seed"])
    T = c["count"]
    bits = [data_bits(rng, n) if n else np.zeros(0, np.uint16) for n in c["sizes"]]
    xs = [to_device(b, dev, o) for b, o in zip(bits, c["xo"])]
    outs = [guarded(n, torch.uint8, dev, o) for n, o in zip(c["sizes"], c["oo"])]
    am = torch.zeros(T, device=dev)
    sc = torch.tensor(c["scales"], dtype=torch.float32, device=dev)
    owner = [0 if (c["shared"] and i % 3 == 0) else i for i in range(T)]
    fp8q.fp8q_multi_quantize_amax(xs, [q for _, q in outs], c["fmt"], [sc[i:i + 1] for i in range(T)],
                                  [am[owner[i]: owner[i] + 1] for i in range(T)])
    torch.cuda.synchronize()
    got_am = am.cpu().numpy()
    want = {}
    for i in range(T):
        rq, ra = par_quantize_amax(bits[i], c["fmt"], np.float32(c["scales"][i]))
        assert_codes_equal(outs[i][1].cpu().numpy(), rq, c["fmt"], f"tensor {i} of {T}")
        check_guards(outs[i][0], c["sizes"][i], c["oo"][i])
        want.setdefault(owner[i], []).append(ra)
    for o, vals in want.items():
        assert_f32_equal([got_am[o]], [combine_amax(vals)], f"amax {o}")


# --------------------------------------------------------------------------- scale update

def draw_update(seed):
    """A random history (1 to ~4700 rows, 1 to ~1200 slots), its specials, the options."""
    rng = np.random.default_rng(seed)
    H = max(1, int(2.0 ** rng.uniform(0, 12.2)))
    S = max(1, int(2.0 ** rng.uniform(0, 10.2)))
    return dict(H=H, S=S, algo=int(rng.integers(2)), fmt=E4M3FN if rng.random() < 0.5 else E5M2,
                margin=int(rng.choice([-64, -3, -1, 0, 0, 1, 2, 7, 64])), per_slot=rng.random() < 0.5,
                steps=int(rng.integers(1, 4)), offset=int(rng.random() < 0.2), data_seed=seed * 7 + 5)


def update_inputs(c):
    """lognormal history and new amaxes with 5% zeros and a few specials (NaN, inf, negative,
    subnormal, near the float32 top), scales from 2^U(-10, 10), slot formats with a few
    unknown codes (whose slots keep their scales)."""
    rng = np.random.default_rng(c["data_seed"])
    H, S = c["H"], c["S"]
    sigma = rng.uniform(0.5, 4.0)
    hist = np.exp(rng.normal(0, sigma, (H, S))).astype(np.float32)
    new = np.exp(rng.normal(0, sigma, S)).astype(np.float32)
    hist[rng.random((H, S)) < 0.05] = 0.0
    new[rng.random(S) < 0.05] = 0.0
    specials = np.array([np.nan, np.inf, -1.5, 1e-45, 3e38, 0.0], np.float32)
    for arr in (hist.reshape(-1), new):
        k = int(rng.integers(0, 4))
        arr[rng.integers(0, arr.size, k)] = specials[rng.integers(0, specials.size, k)]
    scale0 = (2.0 ** rng.uniform(-10, 10, S)).astype(np.float32)
    sf = None
    if c["per_slot"]:
        sf = rng.integers(0, 2, S).astype(np.uint8)
        sf[rng.random(S) < 0.05] = 7
    return hist, new, scale0, sf


UPDATE_CASES = [draw_update(5000 + i) for i in range(24)]


def update_id(c):
    return f"{c['H']}x{c['S']}-a{c['algo']}-f{c['fmt']}-m{c['margin']}-p{int(c['per_slot'])}-o{c['offset']}"


@pytest.mark.parametrize("c", UPDATE_CASES, ids=update_id)
def test_random_scale_update(dev, c):
    hist, new, scale0, sf = update_inputs(c)
    _update_case(dev, hist, new, fmt=c["fmt"], algo=c["algo"], margin=c["margin"], slot_format=sf,
                 steps=c["steps"], scale0=scale0, hist_offset=c["offset"])


@pytest.mark.parametrize("c", UPDATE_CASES, ids=update_id)
def test_random_ring_update(dev, c):
    hist, new, scale0, sf = update_inputs(c)
    rng = np.random.default_rng(c["data_seed"] + 1)
    head = rng.integers(0, c["H"], c["S"]).astype(np.int32)
    bad = rng.random(c["S"]) < 0.05          # corrupt heads: those slots stay untouched
    head[bad] = rng.choice(np.array([-1, c["H"], 1 << 30], np.int32), int(bad.sum()))
    _ring_case(dev, hist, head, new, algo=c["algo"], margin=c["margin"], slot_format=sf,
               steps=c["steps"], scale0=scale0, hist_offset=c["offset"])


def draw_fused(seed):
    rng = np.random.default_rng(seed)
    H = max(1, int(2.0 ** rng.uniform(0, 11)))
    S = max(1, int(2.0 ** rng.uniform(0, 10.2)))
    n = 0 if rng.random() < 0.1 else draw_size(rng, 23)
    return dict(H=H, S=S, slot=int(rng.integers(S)), n=n, algo=int(rng.integers(2)),
                margin=int(rng.choice([-3, 0, 0, 1, 5])), per_slot=rng.random() < 0.5,
                steps=int(rng.integers(1, 4)), seed=seed)


FUSED_CASES = [draw_fused(6000 + i) for i in range(16)]


@pytest.mark.parametrize("c", FUSED_CASES, ids=lambda c: f"{c['H']}x{c['S']}-slot{c['slot']}-n{c['n']}")
def test_random_ring_update_quantize(dev, c):
    """The ring update of every slot fused with the quantize of x by one slot's new scale,
    chained over 1 to 3 steps, against the oracle's update followed by its quantize."""
    _fused_case(dev, c["H"], c["S"], c["slot"], c["n"], c["algo"], c["margin"], c["per_slot"],
                steps=c["steps"], seed=c["seed"])


def test_tensor_list_built_once_gives_the_same_as_the_sequences(dev):
    """A TensorList reused over calls: the same codes and amaxes as passing the sequences."""
    rng = np.random.default_rng(77)
    sizes = [int(v) for v in rng.integers(1, 70000, 300)]
    xs = [to_device(data_bits(rng, n), dev, 0) for n in sizes]
    qa = [torch.empty(n, dtype=torch.uint8, device=dev) for n in sizes]
    qb = [torch.empty(n, dtype=torch.uint8, device=dev) for n in sizes]
    sc = torch.tensor([draw_scale(rng) for _ in sizes], dtype=torch.float32, device=dev)
    am_a, am_b = torch.zeros(len(sizes), device=dev), torch.zeros(len(sizes), device=dev)
    sl = [sc[i:i + 1] for i in range(len(sizes))]
    fp8q.fp8q_multi_quantize_amax(xs, qa, E5M2, sl, [am_a[i:i + 1] for i in range(len(sizes))])
    tl = fp8q.TensorList(xs, qb, sl, [am_b[i:i + 1] for i in range(len(sizes))])
    for _ in range(3):                       # reused: amax max-accumulates to the same values
        fp8q.fp8q_multi_quantize_amax(tl, fmt=E5M2)
    torch.cuda.synchronize()
    for a, b in zip(qa, qb):
        assert torch.equal(a, b)
    assert torch.equal(am_a.view(torch.int32), am_b.view(torch.int32))
    with pytest.raises(ValueError):
        fp8q.fp8q_multi_quantize_amax(tl, qa, E5M2)
