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
