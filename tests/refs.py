"""Independent references used to pin the oracle (test-only).

Nothing here re-types the oracle's loops: values come from library routines
(torch's dtype conversions and ``scaled_dot_product_attention``), applied to
the *logical* per-request K/V arrays the input generator kept before it wrote
them into shuffled pages -- so no page-table arithmetic is involved at all.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F


def bf16_bits_to_f64(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double()


def e4m3_dequant_f64(codes: np.ndarray, scale: float) -> torch.Tensor:
    """(code as float8_e4m3fn -> float32) * scale (float32), then to bfloat16:
    the dequantisation written on the prefix-prefill page, done by torch."""
    f = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).float()
    return (f * torch.tensor(scale, dtype=torch.float32)).to(torch.bfloat16).double()


def logical_kv_f64(p, b):
    if p.kv_dtype == "fp8_e4m3":
        ks = p.k_scale if p.k_scales is None else float(p.k_scales[b])
        vs = p.v_scale if p.v_scales is None else float(p.v_scales[b])
        return e4m3_dequant_f64(p.logical_k[b], ks), e4m3_dequant_f64(p.logical_v[b], vs)
    return bf16_bits_to_f64(p.logical_k[b]), bf16_bits_to_f64(p.logical_v[b])


def sdpa_with_lse(q, k, v, keep, scale):
    """softmax attention by torch SDPA (float64, GQA by ``enable_gqa``).

    q [n, Hq, D], k/v [L, Hkv, D], keep [n, L] bool.  The LSE is recovered
    through one extra key of additive score ``c`` whose value is a unit vector
    in an extra output column: that column equals e^c / (e^c + Z), so
    Z = e^c (1/w - 1).  Returns (O [n, Hq, D], LSE [n, Hq]).
    """
    n, Hq, D = q.shape
    L, Hkv, _ = k.shape
    c = float(np.log(max(L, 1)))
    K = torch.cat([k, torch.zeros(1, Hkv, D, dtype=k.dtype)], 0)
    Vx = torch.zeros(L + 1, Hkv, D + 1, dtype=v.dtype)
    Vx[:L, :, :D] = v
    Vx[L, :, D] = 1.0
    mask = torch.full((n, L + 1), float("-inf"), dtype=torch.float64)
    mask[:, :L][torch.as_tensor(keep)] = 0.0
    mask[:, L] = c
    out = F.scaled_dot_product_attention(
        q.permute(1, 0, 2)[None], K.permute(1, 0, 2)[None], Vx.permute(1, 0, 2)[None],
        attn_mask=mask[None, None], scale=scale, enable_gqa=True)[0].permute(1, 0, 2)
    w = out[..., D]
    Z = np.exp(c) * (1.0 / w - 1.0)
    O = out[..., :D] * ((np.exp(c) + Z) / Z)[..., None]
    return O, torch.log(Z)


def lower_right_causal(n: int, L: int) -> torch.Tensor:
    """Bottom-right-aligned causal mask (query i of n sees keys <= L-n+i),
    the alignment of torch's ``causal_lower_right`` bias."""
    return torch.ones(n, L, dtype=torch.bool).tril(diagonal=L - n)
