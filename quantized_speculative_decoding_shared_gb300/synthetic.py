"""Seeded synthetic inputs for the QSPEC hot path.

This module only draws random inputs of the right shapes and distributions.
It holds none of the method's arithmetic (no quantisation, no softmax, no
acceptance rule), so the CUDA path and the CPU oracle can both be fed from
it without sharing any computation.

Draft tokens are drawn from the draft logits with the Gumbel-max trick
(argmax of logits plus Gumbel noise), which samples the softmax of the
logits without computing it.

Shapes follow the layer sizes the workloads name:
  Llama-3-8B:  hidden 4096, q 4096, k/v 1024, inter 14336, vocab 128256,
               32 layers, 8 KV heads x 128.
  Qwen2.5-7B:  hidden 3584, q 3584, k/v 512, inter 18944, vocab 152064,
               28 layers, 4 KV heads x 128.
"""
from __future__ import annotations

import numpy as np
import torch

GROUP = 128

LLAMA3_8B = dict(hidden=4096, q=4096, kv=1024, inter=14336, vocab=128256, layers=32,
                 kv_heads=8, head_dim=128)
QWEN25_7B = dict(hidden=3584, q=3584, kv=512, inter=18944, vocab=152064, layers=28,
                 kv_heads=4, head_dim=128)


def layer_linears(shape: dict) -> list[tuple[str, int, int]]:
    """(name, N, K) of the seven linears of one decoder layer."""
    h, q, kv, it = shape["hidden"], shape["q"], shape["kv"], shape["inter"]
    return [("q_proj", q, h), ("k_proj", kv, h), ("v_proj", kv, h), ("o_proj", h, q),
            ("gate_proj", it, h), ("up_proj", it, h), ("down_proj", h, it)]


def fused_layer_linears(shape: dict) -> list[tuple[str, int, int]]:
    """The same seven linears with the ones that share an input stacked along N:
    q/k/v (one input) and gate/up (one input).  Same bytes and flops."""
    h, q, kv, it = shape["hidden"], shape["q"], shape["kv"], shape["inter"]
    return [("qkv_proj", q + 2 * kv, h), ("o_proj", h, q), ("gate_up_proj", 2 * it, h),
            ("down_proj", h, it)]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def weights(N: int, K: int, seed: int, device="cpu", s_lo=0.005, s_hi=0.02):
    """INT4 codes uniform in [0, 15], fp16 scales U(s_lo, s_hi), zero points
    uniform integers in [0, 15] stored as fp16.

    Returns (codes uint8 [N][K], s fp16 [N][K/128], z fp16 [N][K/128])."""
    assert K % GROUP == 0
    g = _gen(seed, device)
    G = K // GROUP
    codes = torch.randint(0, 16, (N, K), generator=g, device=device, dtype=torch.uint8)
    s = (torch.rand((N, G), generator=g, device=device) * (s_hi - s_lo) + s_lo).to(torch.float16)
    z = torch.randint(0, 16, (N, G), generator=g, device=device).to(torch.float16)
    return codes, s, z


def activations(M: int, K: int, seed: int, device="cpu", outlier_frac=0.0, outlier_scale=20.0,
                std=1.0):
    """bf16 [M][K] N(0, std^2); a fixed set of K channels (chosen by the seed)
    is multiplied by outlier_scale for every row."""
    g = _gen(seed, device)
    x = torch.randn((M, K), generator=g, device=device) * std
    n_out = int(round(outlier_frac * K))
    if n_out:
        ch = torch.randperm(K, generator=g, device=device)[:n_out]
        x[:, ch] *= outlier_scale
    return x.to(torch.bfloat16)


def gumbel_argmax(logits: torch.Tensor, g: torch.Generator) -> torch.Tensor:
    """One sample per row of softmax(logits) by the Gumbel-max trick."""
    u = torch.rand(logits.shape, generator=g, device=logits.device, dtype=torch.float64)
    u = u.clamp_min(1e-300)
    gum = -torch.log(-torch.log(u))
    return torch.argmax(logits.double() + gum, dim=-1).to(torch.int32)


def logits_shared_offset(B: int, gamma: int, V: int, seed: int, device="cpu", std=2.0):
    """Target and draft logits N(0, std^2) plus one N(0, 1) offset per
    vocabulary id shared by both; drafts drawn from the draft rows.

    Returns P bf16 [B][gamma+1][V], Q bf16 [B][gamma][V], drafts int32 [B][gamma]."""
    g = _gen(seed, device)
    c = torch.randn((V,), generator=g, device=device)
    P = torch.randn((B, gamma + 1, V), generator=g, device=device) * std + c
    Q = torch.randn((B, gamma, V), generator=g, device=device) * std + c
    P, Q = P.to(torch.bfloat16), Q.to(torch.bfloat16)
    drafts = gumbel_argmax(Q.float(), g)
    return P, Q, drafts


def logits_noisy_draft(B: int, gamma: int, V: int, seed: int, device="cpu", p_std=3.0,
                       q_noise=0.5):
    """Target logits N(0, p_std^2); draft logits = target + N(0, q_noise^2)
    on the first gamma rows; drafts drawn from the draft rows."""
    g = _gen(seed, device)
    Pf = torch.randn((B, gamma + 1, V), generator=g, device=device) * p_std
    Qf = Pf[:, :gamma, :] + torch.randn((B, gamma, V), generator=g, device=device) * q_noise
    P, Q = Pf.to(torch.bfloat16), Qf.to(torch.bfloat16)
    drafts = gumbel_argmax(Q.float(), g)
    return P, Q, drafts


def kv_cache(L: int, B: int, H: int, T: int, D: int, seed: int, device="cpu"):
    """K and V caches bf16 [L][B][H][T][D] filled N(0, 1)."""
    g = _gen(seed, device)
    k = torch.randn((L, B, H, T, D), generator=g, device=device).to(torch.bfloat16)
    v = torch.randn((L, B, H, T, D), generator=g, device=device).to(torch.bfloat16)
    return k, v


def kv_new(L: int, B: int, gamma: int, H: int, D: int, seed: int, device="cpu"):
    """Verify-pass K and V rows bf16 [L][B][gamma+1][H][D] filled N(0, 1)."""
    g = _gen(seed, device)
    k = torch.randn((L, B, gamma + 1, H, D), generator=g, device=device).to(torch.bfloat16)
    v = torch.randn((L, B, gamma + 1, H, D), generator=g, device=device).to(torch.bfloat16)
    return k, v


def base_positions(B: int, T: int, gamma: int, seed: int, device="cpu"):
    """Per-sequence cache position of the last confirmed token, uniform in
    [0, T - gamma - 2] so that every accepted row fits."""
    g = _gen(seed, device)
    return torch.randint(0, T - gamma - 1, (B,), generator=g, device=device, dtype=torch.int32)


# ---------------------------------------------------------------------------
# bit-pattern views used to hand tensors to the oracle (numpy, host)
# ---------------------------------------------------------------------------
def bits16(t: torch.Tensor) -> np.ndarray:
    """bf16 / fp16 tensor -> uint16 numpy array of its bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bits_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
