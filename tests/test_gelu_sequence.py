"""The GELU producer's fixed binary32 sequence (tests/csrc/gelu_sequence.c, the
arithmetic both GELU kernels follow) meets the tolerance stated against the
float64 definition, on every bf16 input.  This checks, on the CPU, that the
tolerance derived for that arithmetic actually holds for it; the GPU tests then
hold the kernels to the same tolerance and to these bits."""
import numpy as np


def test_sequence_within_the_gelu_tolerance_for_every_bf16_input(orc, seq_gelu):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    y = seq_gelu(h)
    r = orc.gelu_ref_array(h)
    x = (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    E = orc.gelu_tolerance(x, r)
    ok = orc.bf16_within(y, r, E)
    assert ok.all(), f"{(~ok).sum()} inputs outside, first {h[~ok][:5]}"
    # and the sequence is the float64 value rounded once to bf16 for nearly every input
    big = np.isfinite(x) & (np.abs(r) >= orc.GELU_TINY)
    assert np.mean((y == orc.f64_to_bf16_array(r))[big]) > 0.99


def test_sequence_is_monotone_from_zero_and_small_for_negative_inputs(seq_gelu):
    """The two facts the codes-only table kernel takes its amax from (the largest input of a
    thread gives the largest |y|, unless it is below about 0.3): from +0 to +inf y never
    decreases and is not negative, and every negative input (-0 to -inf) gives |y| < 0.1875."""
    pos = np.arange(0x0000, 0x7F81, dtype=np.uint32).astype(np.uint16)  # +0 ... +inf, in value order
    yp = (seq_gelu(pos).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert not np.isnan(yp).any() and (yp >= 0).all()
    assert (np.diff(yp) >= 0).all()
    assert yp[-1] == np.inf
    neg = np.arange(0x8000, 0xFF81, dtype=np.uint32).astype(np.uint16)  # -0 ... -inf
    yn = np.abs((seq_gelu(neg).astype(np.uint32) << 16).view(np.float32).astype(np.float64))
    assert (yn < 0.1875).all()
    assert 0.16 < yn.max() < 0.172            # GELU's minimum, about -0.170 near x = -0.75
    # the smallest input whose y reaches the bound: inputs below it send a thread to its re-read
    first = pos[np.argmax(yp >= 0.1875)]
    x = float((np.uint32(first) << 16).view(np.float32))
    assert 0.25 < x < 0.35
