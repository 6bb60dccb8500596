"""Seeded synthetic inputs for KDA -- shared by the tests, the benchmark and
the smoke check. Holds none of the operator's arithmetic: it only draws
random numbers with the distributions of the workloads and casts them to the
stored dtypes. Both the CUDA path and the oracle consume exactly the values
returned here.

Recipe (per token t, head h):
  q, k  ~ N(0, 1) per channel, then L2-normalised over the head dim (fp32),
          then cast to the I/O dtype;
  v     ~ N(0, 1), cast to the I/O dtype;
  beta  = sigmoid(N(0, 1)), cast to the I/O dtype;
  g     = -5 * sigmoid(N(0, 1)) per channel, kept fp32      ("standard"),
          or -5 + 0.5 * sigmoid(N(0, 1))                     ("floor");
  initial state: zeros, or N(0, 0.02^2) fp32.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

D_HEAD = 128


def _dtype(io: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[io]


@dataclass
class PrefillInputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    init_state: Optional[torch.Tensor]
    cu_seqlens: Optional[torch.Tensor]  # int32 [N+1] (None: one sequence)
    scale: float
    lens: list = field(default_factory=list)

    @property
    def T_total(self) -> int:
        return self.q.shape[0]

    @property
    def H(self) -> int:
        return self.q.shape[1]

    @property
    def N(self) -> int:
        return len(self.lens)


def _normal(gen, shape, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def _l2norm(x):
    return x / torch.linalg.vector_norm(x, dim=-1, keepdim=True).clamp_min(1e-6)


def token_block(gen, T, H, D, io, g_mode, device):
    """Draw T tokens x H heads (q, k, v, g, beta) from one generator."""
    dt = _dtype(io)
    q = _l2norm(_normal(gen, (T, H, D), device)).to(dt)
    k = _l2norm(_normal(gen, (T, H, D), device)).to(dt)
    v = _normal(gen, (T, H, D), device).to(dt)
    beta = torch.sigmoid(_normal(gen, (T, H), device)).to(dt)
    z = torch.sigmoid(_normal(gen, (T, H, D), device))
    if g_mode == "standard":
        g = -5.0 * z
    elif g_mode == "floor":
        g = -5.0 + 0.5 * z
    else:
        raise ValueError(g_mode)
    return q, k, v, g.contiguous(), beta


def prefill_inputs(lens, H, io="bf16", seed=0, g_mode="standard", init="zero", D=D_HEAD,
                   device="cpu", block_tokens=1 << 14):
    """Packed prefill inputs for sequences of the given lengths.

    Sequence n draws from its own generator seeded (seed * 1_000_003 + n), in
    blocks of `block_tokens` tokens, so any sequence can be regenerated alone
    (``sequence_inputs``) and large workloads are produced without a large
    fp32 temporary."""
    lens = [int(x) for x in lens]
    T = sum(lens)
    dt = _dtype(io)
    q = torch.empty((T, H, D), dtype=dt, device=device)
    k = torch.empty_like(q)
    v = torch.empty_like(q)
    g = torch.empty((T, H, D), dtype=torch.float32, device=device)
    beta = torch.empty((T, H), dtype=dt, device=device)
    off = 0
    for n, L in enumerate(lens):
        gen = torch.Generator(device=device)
        gen.manual_seed(seed * 1_000_003 + n)
        done = 0
        while done < L:
            b = min(block_tokens, L - done)
            qq, kk, vv, gg, bb = token_block(gen, b, H, D, io, g_mode, device)
            sl = slice(off + done, off + done + b)
            q[sl], k[sl], v[sl], g[sl], beta[sl] = qq, kk, vv, gg, bb
            done += b
        off += L
    init_state = None
    if init == "normal":
        gen = torch.Generator(device=device)
        gen.manual_seed(seed * 1_000_003 + 999_983)
        init_state = 0.02 * _normal(gen, (len(lens), H, D, D), device)
    elif init != "zero":
        raise ValueError(init)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    return PrefillInputs(q, k, v, g, beta, init_state, cu.to(device), D ** -0.5, lens)


def sequence_inputs(lens, n, H, io="bf16", seed=0, g_mode="standard", D=D_HEAD, device="cpu",
                    block_tokens=1 << 14):
    """Regenerate sequence n of ``prefill_inputs(lens, ...)`` on its own."""
    L = int(lens[n])
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 1_000_003 + n)
    parts = []
    done = 0
    while done < L:
        b = min(block_tokens, L - done)
        parts.append(token_block(gen, b, H, D, io, g_mode, device))
        done += b
    return tuple(torch.cat([p[i] for p in parts]) for i in range(5))


def varlen_lengths(n_seqs=64, lo=1024, hi=32768, seed=4):
    gen = torch.Generator()
    gen.manual_seed(seed)
    return torch.randint(lo, hi + 1, (n_seqs,), generator=gen).tolist()


def decode_inputs(B, H, steps, io="bf16", seed=2, D=D_HEAD, device="cpu"):
    """Per-step decode inputs [steps, B, H, ...] and an N(0, 0.02^2) state."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    q, k, v, g, beta = token_block(gen, steps * B, H, D, io, "standard", device)
    shp = (steps, B, H, D)
    state = 0.02 * _normal(gen, (B, H, D, D), device)
    return (q.view(shp), k.view(shp), v.view(shp), g.view(shp), beta.view(steps, B, H),
            state, D ** -0.5)


# The five workloads, named by what they are.
WORKLOADS = {
    "tiny_f32": dict(lens=[64], H=2, io="f32", chunk=16, g_mode="standard", init="zero", seed=1000),
    "prefill_mid_bf16": dict(lens=[8192], H=32, io="bf16", chunk=64, g_mode="standard", init="zero",
                             seed=1001),
    "decode_b256_h96": dict(B=256, H=96, steps=64, io="bf16", seed=1002),
    "append_h96": dict(prior=32768, T=65536, H=96, io="bf16", chunk=64, g_mode="standard",
                       seed=1003),
    "varlen64_h32_floor": dict(n_seqs=64, lo=1024, hi=32768, H=32, io="bf16", chunk=64,
                               g_mode="floor", init="normal", seed=1004),
}
