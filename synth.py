"""Seeded synthetic inputs for the PACE decode path.

This module is the only code shared by the CUDA-path tests/benchmark and the CPU oracle. It holds
none of the method's arithmetic: it draws random tensors and shapes them like the pages' workloads.

Recipe (every workload):
  * q, k ~ N(0, 1) per element, then L2-normalised over d_k per (sequence, head, token);
  * v ~ N(0, 1), with a few value channels per head scaled x8 for every token and sequence
    (persistent column outliers, the structure [P2] "3. Method & Key Results", Figure 3 describes);
    the channels are drawn once per (layer, head) from the seed;
  * a_t ~ U[a_lo, a_hi] per (sequence, head, token), or one a_h per head for every token when
    ``a_per_head`` is set (the "mean decay" workload);
  * beta_t = sigmoid(N(0, 1));
  * with bf16 I/O, q, k and v are rounded to bf16 (nearest, ties to even) before anyone reads them.

Random numbers come from numpy's counter-based Philox-4x32-10 generator, keyed by
(seed, tensor, layer, token), so any token of any layer can be regenerated on its own.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np

_T_Q, _T_K, _T_V, _T_A, _T_B, _T_OUT, _T_AH = 1, 2, 3, 4, 5, 6, 7


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    d_k: int
    d_v: int
    seed: int
    n_outliers: int = 4
    outlier_scale: float = 8.0
    a_lo: float = 0.90
    a_hi: float = 0.999
    a_per_head: bool = False
    io: str = "bf16"            # "bf16" or "f32"
    layers: int = 1
    prefill: int = 512
    decode: int = 256
    dP: int = 8
    g: int = 64
    zero_point: int = 0
    mixed_buffer: bool = False
    int8_heads: int = 0         # heads kept at 8 bits (chosen by the E_h ranking)
    batches: tuple = field(default=())

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five synthetic workloads (shapes and distributions as stated for each).
WORKLOADS = {
    # Tiny PACE-4: 1 layer, 2 heads, d=64, batch 2, one 256-token chunk then 64 decode tokens.
    "tiny": Workload("tiny", B=2, H=2, d_k=64, d_v=64, seed=0, n_outliers=3, io="f32",
                     prefill=256, decode=64),
    # PACE-4 decode: 32 heads, d=128, batch 64, 512-token context, 256 decode tokens.
    "pace4": Workload("pace4", B=64, H=32, d_k=128, d_v=128, seed=1),
    # PACE-4/8: g=32 zero-point, 8 of 32 heads int8, mixed buffer, per-head decay.
    "pace48": Workload("pace48", B=128, H=32, d_k=128, d_v=128, seed=2, a_lo=0.85, a_hi=0.999,
                       a_per_head=True, g=32, zero_point=1, mixed_buffer=True, int8_heads=8),
    # Batch sweep: 24 layers x 16 heads, 512-token context, 128 decode tokens.
    "sweep": Workload("sweep", B=16, H=16, d_k=128, d_v=128, seed=3, layers=24, decode=128,
                      batches=(1, 2, 4, 8, 16, 32, 64, 128)),
    # Long context: 48 heads, batch 16, 32,768-token prefill, 1,024 decode tokens, slow decay.
    "longctx": Workload("longctx", B=16, H=48, d_k=128, d_v=128, seed=4, a_lo=0.95, a_hi=0.9999,
                        prefill=32768, decode=1024),
}


def workload(name: str, **overrides) -> Workload:
    wl = WORKLOADS[name]
    return wl.with_(**overrides) if overrides else wl


def _rng(seed: int, tensor: int, layer: int, t: int) -> np.random.Generator:
    key = np.array([seed & 0xFFFFFFFFFFFFFFFF,
                    (tensor << 56) | ((layer & 0xFFFF) << 40) | (t & 0xFFFFFFFFFF)], dtype=np.uint64)
    return np.random.Generator(np.random.Philox(key=key))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even) using torch's conversion; fp32 result."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).to(torch.float32).numpy()


def outlier_channels(wl: Workload, layer: int = 0) -> np.ndarray:
    """[H, n_outliers] value channels scaled up for every token of that head."""
    out = np.zeros((wl.H, wl.n_outliers), np.int64)
    for h in range(wl.H):
        out[h] = np.sort(_rng(wl.seed, _T_OUT, layer, h).choice(wl.d_v, wl.n_outliers, replace=False))
    return out


def head_decays(wl: Workload, layer: int = 0) -> np.ndarray:
    """[H] per-head decay a_h for workloads that hold a_t = a_h for every token."""
    return _rng(wl.seed, _T_AH, layer, 0).uniform(wl.a_lo, wl.a_hi, wl.H).astype(np.float32)


def token_inputs(wl: Workload, t: int, layer: int = 0) -> dict:
    """Inputs of token position t for all sequences and heads.

    Returns q, k [B, H, d_k], v [B, H, d_v], a, beta [B, H], all fp32 (bf16-exact when io == "bf16").
    """
    B, H = wl.B, wl.H
    q = _rng(wl.seed, _T_Q, layer, t).standard_normal((B, H, wl.d_k))
    k = _rng(wl.seed, _T_K, layer, t).standard_normal((B, H, wl.d_k))
    v = _rng(wl.seed, _T_V, layer, t).standard_normal((B, H, wl.d_v))
    q /= np.sqrt(np.einsum("...i,...i->...", q, q))[..., None]
    k /= np.sqrt(np.einsum("...i,...i->...", k, k))[..., None]
    ch = outlier_channels(wl, layer)
    for h in range(H):
        v[:, h, ch[h]] *= wl.outlier_scale
    if wl.a_per_head:
        a = np.broadcast_to(head_decays(wl, layer)[None, :], (B, H)).copy()
    else:
        a = _rng(wl.seed, _T_A, layer, t).uniform(wl.a_lo, wl.a_hi, (B, H))
    beta = 1.0 / (1.0 + np.exp(-_rng(wl.seed, _T_B, layer, t).standard_normal((B, H))))
    q, k, v = (x.astype(np.float32) for x in (q, k, v))
    if wl.io == "bf16":
        q, k, v = round_bf16(q), round_bf16(k), round_bf16(v)
    return {"q": q, "k": k, "v": v, "a": a.astype(np.float32), "beta": beta.astype(np.float32)}


def chunk_inputs(wl: Workload, t0: int, n: int, layer: int = 0) -> dict:
    """Tokens t0 .. t0+n-1 stacked on axis 2: q, k [B, H, n, d_k], v [B, H, n, d_v], a, beta [B, H, n]."""
    out = None
    for i in range(n):
        tk = token_inputs(wl, t0 + i, layer)
        if out is None:
            out = {key: np.empty(val.shape[:2] + (n,) + val.shape[2:], np.float32) for key, val in tk.items()}
        for key, val in tk.items():
            out[key][:, :, i] = val
    return out


def device_chunk_inputs(wl: Workload, t0: int, n: int, layer: int = 0, device="cuda") -> dict:
    """The same recipe drawn on the device with torch's Philox generator (seeded by workload seed, layer
    and first token), for benchmarks that need many tokens quickly and no oracle comparison.
    Returns torch tensors: q, k, v [B, H, n, d] in the I/O dtype, a, beta [B, H, n] fp32."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed((wl.seed * 1_000_003 + layer * 65_537 + t0) & 0x7FFFFFFFFFFFFFFF)
    B, H = wl.B, wl.H
    q = torch.randn(B, H, n, wl.d_k, generator=g, device=device)
    k = torch.randn(B, H, n, wl.d_k, generator=g, device=device)
    v = torch.randn(B, H, n, wl.d_v, generator=g, device=device)
    q = q / q.norm(dim=-1, keepdim=True)
    k = k / k.norm(dim=-1, keepdim=True)
    ch = torch.from_numpy(outlier_channels(wl, layer)).to(device)
    scale = torch.ones(H, wl.d_v, device=device)
    scale.scatter_(1, ch, wl.outlier_scale)
    v = v * scale[None, :, None, :]
    if wl.a_per_head:
        a = torch.from_numpy(head_decays(wl, layer)).to(device)[None, :, None].expand(B, H, n).contiguous()
    else:
        a = torch.rand(B, H, n, generator=g, device=device) * (wl.a_hi - wl.a_lo) + wl.a_lo
    beta = torch.sigmoid(torch.randn(B, H, n, generator=g, device=device))
    dt = torch.bfloat16 if wl.io == "bf16" else torch.float32
    return {"q": q.to(dt).contiguous(), "k": k.to(dt).contiguous(), "v": v.to(dt).contiguous(),
            "a": a.float().contiguous(), "beta": beta.float().contiguous()}
