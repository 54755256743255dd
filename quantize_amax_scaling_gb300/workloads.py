"""Seeded synthetic inputs shaped like the workloads the FP8 pages describe.

This module only draws random numbers; it holds none of the quantization,
amax or scale arithmetic, so both the CUDA path and the CPU oracle can be fed
from it.  Every generator takes an explicit seed and a torch device; draws are
made with a ``torch.Generator`` on that device, so the same seed on the same
device gives the same bytes.  Parity tests copy device-drawn inputs to the host
for the oracle, so the two sides always see identical bits.

Shapes follow the MLP in "Fusion of Fp8 quantization and amax reduction
kernels" (openxla/xla issue, reproducer ``test.py``: sequence 2048, batch 4,
hidden 4096, FFN 16384, bf16) and the 96-layer stack behind "Implement fused
kernel for FP8 scale update" (TransformerEngine PR): 6 FP8 meta slots per
layer, amax history length 1024.
"""
from __future__ import annotations

import math

import torch

# Per-config seeds: config k uses 1000 + k; a "previous step" draw uses seed + 1.
SEED_TINY = 1001
SEED_MLP = 1002
SEED_FFN = 1003
SEED_GRAD = 1004
SEED_UPDATE = 1005

HIDDEN = 4096
SEQ = 2048
BATCH = 4
FFN = 16384
LAYERS = 96
SLOTS_PER_LAYER = 6
HISTORY_LEN = 1024

# Twelve ragged tensors from 2048x12288 up to 12288x4096.
RAGGED_SHAPES = [
    (2048, 12288), (2048, 16384), (3072, 12288), (4096, 8192),
    (4096, 12288), (6144, 4096), (6144, 6144), (8192, 4096),
    (8192, 6144), (10240, 4096), (11264, 4096), (12288, 4096),
]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def uniform_bf16(shape, seed: int, device="cpu") -> torch.Tensor:
    """U[0,1) in float32, stored as bf16 (the page-2 JAX example's A and B)."""
    g = _gen(seed, device)
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def tiny_pair(device="cpu"):
    """A (16x32) and B (32x64), bf16 U[0,1)."""
    return (uniform_bf16((16, 32), SEED_TINY, device),
            uniform_bf16((32, 64), SEED_TINY + 100, device))


def mlp_activation(seed: int = SEED_MLP, device="cpu", shape=(SEQ * BATCH, HIDDEN),
                   outlier_frac: float = 1e-3, outlier_gain: float = 100.0) -> torch.Tensor:
    """N(0,1) bf16 with a uniformly chosen 0.1% of entries multiplied by 100."""
    g = _gen(seed, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    n = x.numel()
    k = max(1, int(n * outlier_frac))
    idx = torch.randint(0, n, (k,), generator=g, device=device)
    flat = x.view(-1)
    flat[idx] = flat[idx] * outlier_gain
    return x.to(torch.bfloat16)


def gelu_activation(seed: int = SEED_FFN, device="cpu", shape=(SEQ * BATCH, FFN)) -> torch.Tensor:
    """gelu(N(0,1)) (tanh form), computed in float32 and stored as bf16."""
    g = _gen(seed, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return torch.nn.functional.gelu(x, approximate="tanh").to(torch.bfloat16)


def residual_stream(seed: int = SEED_MLP + 7, device="cpu", shape=(SEQ * BATCH, HIDDEN),
                    outlier_frac: float = 1e-3, outlier_gain: float = 100.0) -> torch.Tensor:
    """LayerNorm input: row r is N(mu_r, sigma_r^2) with mu_r ~ U(-2, 2) and
    sigma_r ~ U(0.5, 4), and a uniformly chosen 0.1% of entries times 100; bf16."""
    g = _gen(seed, device)
    rows = shape[0]
    mu = torch.rand((rows, 1), generator=g, device=device) * 4.0 - 2.0
    sigma = torch.rand((rows, 1), generator=g, device=device) * 3.5 + 0.5
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * sigma + mu
    n = x.numel()
    k = max(1, int(n * outlier_frac))
    idx = torch.randint(0, n, (k,), generator=g, device=device)
    flat = x.view(-1)
    flat[idx] = flat[idx] * outlier_gain
    return x.to(torch.bfloat16)


def layernorm_params(hidden: int, seed: int = SEED_MLP + 8, device="cpu"):
    """gamma = 1 + 0.1 N(0,1) and beta = 0.1 N(0,1), float32 [hidden] (a trained-looking
    perturbation of Flax's ones/zeros initialisation)."""
    g = _gen(seed, device)
    gamma = 1.0 + 0.1 * torch.randn(hidden, generator=g, device=device, dtype=torch.float32)
    beta = 0.1 * torch.randn(hidden, generator=g, device=device, dtype=torch.float32)
    return gamma, beta


def truncated_normal_weight(shape, fan_in: int, seed: int, device="cpu") -> torch.Tensor:
    """Normal truncated at +-2 sigma, rescaled to variance 1/fan_in (variance-scaling init)."""
    g = _gen(seed, device)
    lo = 0.5 * (1.0 + math.erf(-2.0 / math.sqrt(2.0)))
    hi = 0.5 * (1.0 + math.erf(2.0 / math.sqrt(2.0)))
    u = torch.rand(shape, generator=g, device=device, dtype=torch.float64)
    z = torch.special.ndtri(lo + u * (hi - lo)).clamp_(-2.0, 2.0)
    # std of a unit normal truncated to [-2, 2]
    trunc_std = 0.87962566103423978
    w = z * (math.sqrt(1.0 / fan_in) / trunc_std)
    return w.to(torch.bfloat16)


def ffn_tensors(device="cpu", seed: int = SEED_FFN, scale_down: int = 1):
    """Activation 8192x16384 = gelu(N(0,1)); W1 4096x16384 and W2 16384x4096.

    ``scale_down`` divides the leading dimension of every tensor (small parity cases).
    """
    act = gelu_activation(seed, device, (SEQ * BATCH // scale_down, FFN))
    w1 = truncated_normal_weight((HIDDEN // scale_down, FFN), HIDDEN, seed + 10, device)
    w2 = truncated_normal_weight((FFN // scale_down, HIDDEN), FFN, seed + 20, device)
    return [act, w1, w2]


def gradient(shape, seed: int, device="cpu", mu: float = -12.0, sigma: float = 3.0,
             zero_frac: float = 0.01, n_inf: int = 8) -> torch.Tensor:
    """sign-random x lognormal(mu, sigma) bf16, with 1% signed zeros and a few +-inf."""
    g = _gen(seed, device)
    mag = torch.exp(torch.randn(shape, generator=g, device=device, dtype=torch.float32) * sigma + mu)
    sign = torch.randint(0, 2, shape, generator=g, device=device, dtype=torch.int8)
    x = torch.where(sign.bool(), -mag, mag)
    flat = x.view(-1)
    n = flat.numel()
    nz = max(1, int(n * zero_frac))
    zi = torch.randint(0, n, (nz,), generator=g, device=device)
    flat[zi] = torch.where(flat[zi] < 0, torch.full_like(flat[zi], -0.0), torch.zeros_like(flat[zi]))
    ii = torch.randint(0, n, (n_inf,), generator=g, device=device)
    infs = torch.tensor([math.inf, -math.inf], device=device).repeat((n_inf + 1) // 2)[:n_inf]
    flat[ii] = infs
    return x.to(torch.bfloat16)


def gradient_tensors(device="cpu", seed: int = SEED_GRAD, scale_down: int = 1):
    """Backward gradients 8192x16384 and 8192x4096 (e5m2 workload)."""
    return [gradient((SEQ * BATCH // scale_down, FFN), seed, device),
            gradient((SEQ * BATCH // scale_down, HIDDEN), seed + 10, device)]


def lognormal_with_zeros(shape, seed: int, device="cpu", sigma: float = 2.0,
                         zero_frac: float = 0.02) -> torch.Tensor:
    """float32 exp(N(0, sigma^2)) with a seeded 2% of entries set to exactly zero."""
    g = _gen(seed, device)
    x = torch.exp(torch.randn(shape, generator=g, device=device, dtype=torch.float32) * sigma)
    flat = x.view(-1)
    n = flat.numel()
    nz = max(1, int(n * zero_frac))
    flat[torch.randint(0, n, (nz,), generator=g, device=device)] = 0.0
    return x


def scale_update_inputs(device="cpu", seed: int = SEED_UPDATE, history_len: int = HISTORY_LEN,
                        num_slots: int = LAYERS * SLOTS_PER_LAYER):
    """History [H][S] and a new amax vector [S], both lognormal(0, 2) with 2% zeros.

    Also returns starting scales of 1.0 and a slot-format vector in which the
    last two of every layer's six slots are e5m2 (code 1), the rest e4m3fn (0).
    """
    hist = lognormal_with_zeros((history_len, num_slots), seed, device)
    amax_new = lognormal_with_zeros((num_slots,), seed + 1, device)
    scale = torch.ones(num_slots, device=device, dtype=torch.float32)
    scale_inv = torch.ones(num_slots, device=device, dtype=torch.float32)
    slot = torch.arange(num_slots, device=device) % SLOTS_PER_LAYER
    slot_format = (slot >= 4).to(torch.uint8)
    return hist, amax_new, scale, scale_inv, slot_format


def ragged_tensors(device="cpu", seed: int = SEED_UPDATE + 50, scale_down: int = 1):
    """Twelve bf16 N(0,1) tensors of the ragged shapes (leading dim divided by scale_down)."""
    out = []
    for i, (r, c) in enumerate(RAGGED_SHAPES):
        g = _gen(seed + i, device)
        out.append(torch.randn((max(1, r // scale_down), c), generator=g, device=device,
                               dtype=torch.float32).to(torch.bfloat16))
    return out


def bf16_bits(t: torch.Tensor):
    """Host numpy uint16 view of a bf16 tensor's bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16").reshape(-1)


def all_bf16_patterns(device="cpu") -> torch.Tensor:
    """Every one of the 65536 bf16 bit patterns, in order."""
    import numpy as np
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.int16)
    return torch.from_numpy(bits.copy()).view(torch.bfloat16).to(device)
