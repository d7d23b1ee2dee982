"""Seeded synthetic inputs for the training-step kernels.

This module only *makes inputs*: parameter tables, initial weights, scaled
16-bit gradients, forward softmax probabilities and the LayerNorm forward's
saved statistics.  It contains none of the backward or optimizer arithmetic,
and it imports neither the CUDA library nor the CPU oracle, so both can be fed
the very same bytes.

Randomness comes from ``torch.Generator`` streams seeded from ``(seed, salt)``;
large inputs are drawn on the device, small ones on the host.  Value recipes:

* AdamW: theta ~ N(0, 0.02) fp32, m = v = 0, gradient = N(0, sigma) *
  loss_scale rounded to the 16-bit gradient dtype (sigma is a standard
  deviation), a fresh draw for every (seed, step).
* Softmax backward: P = row softmax of N(0,1) logits computed in float64 and
  rounded to the I/O dtype; with ``causal_period=S`` (and ``causal_offset=o``)
  row r only sees columns j <= r mod S + o and the masked entries are exactly
  0; dY ~ N(0,1).
* RMSNorm backward: as LayerNorm, with inv_rms = 1/sqrt(mean(x^2) + eps).
* LayerNorm backward: x ~ N(0,1) and dY ~ N(0, dy_std) in the I/O dtype,
  gamma ~ N(1, 0.1) fp32, and the forward's saved mean and inv_std =
  1/sqrt(var + eps) (biased variance) computed in float64 from the stored x
  and rounded to fp32.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Sequence, Tuple

import torch

# ----------------------------------------------------------------------------- tables
def gpt2_small_shapes() -> List[Tuple[str, Tuple[int, ...]]]:
    """GPT-2-small parameter list: 148 tensors, 124,439,808 parameters."""
    d, v, ctx, L = 768, 50257, 1024, 12
    out = [("wte", (v, d)), ("wpe", (ctx, d))]
    for i in range(L):
        p = f"h.{i}."
        out += [
            (p + "ln_1.weight", (d,)), (p + "ln_1.bias", (d,)),
            (p + "attn.c_attn.weight", (d, 3 * d)), (p + "attn.c_attn.bias", (3 * d,)),
            (p + "attn.c_proj.weight", (d, d)), (p + "attn.c_proj.bias", (d,)),
            (p + "ln_2.weight", (d,)), (p + "ln_2.bias", (d,)),
            (p + "mlp.c_fc.weight", (d, 4 * d)), (p + "mlp.c_fc.bias", (4 * d,)),
            (p + "mlp.c_proj.weight", (4 * d, d)), (p + "mlp.c_proj.bias", (d,)),
        ]
    out += [("ln_f.weight", (d,)), ("ln_f.bias", (d,))]
    return out


def llama7b_shapes() -> List[Tuple[str, Tuple[int, ...]]]:
    """Llama-7B parameter list: 291 tensors, 6,738,415,616 parameters."""
    d, ff, v, L = 4096, 11008, 32000, 32
    out = [("embed_tokens", (v, d))]
    for i in range(L):
        p = f"layers.{i}."
        out += [
            (p + "q_proj", (d, d)), (p + "k_proj", (d, d)),
            (p + "v_proj", (d, d)), (p + "o_proj", (d, d)),
            (p + "gate_proj", (ff, d)), (p + "up_proj", (ff, d)),
            (p + "down_proj", (d, ff)),
            (p + "input_layernorm", (d,)), (p + "post_attention_layernorm", (d,)),
        ]
    out += [("norm", (d,)), ("lm_head", (v, d))]
    return out


def numel(shape: Sequence[int]) -> int:
    n = 1
    for s in shape:
        n *= int(s)
    return n


def _gen(device, seed: int, salt: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 0x9E3779B1 + int(salt) * 0x85EBCA77 + 0x165667B1) % (2**63))
    return g


# ----------------------------------------------------------------------------- AdamW
ARENA_ALIGN = 128  # elements; tensors start on 512-byte (fp32) / 256-byte (16-bit) boundaries


@dataclass
class AdamWState:
    """Flat arenas (one per buffer kind) and per-tensor views into them."""
    names: List[str]
    sizes: List[int]
    offsets: List[int]
    theta: torch.Tensor          # fp32 arena
    m: torch.Tensor              # fp32 arena
    v: torch.Tensor              # fp32 arena
    grad: torch.Tensor           # 16-bit arena (bf16 or fp16)
    copy: torch.Tensor           # 16-bit arena (bf16 or fp16)
    grad_std: float
    loss_scale: float
    seed: int
    views: dict = field(default_factory=dict)

    @property
    def n_params(self) -> int:
        return sum(self.sizes)

    def tensor(self, kind: str, i: int) -> torch.Tensor:
        a = getattr(self, kind)
        return a.narrow(0, self.offsets[i], self.sizes[i])


def layout(sizes: Sequence[int], align: int = ARENA_ALIGN) -> Tuple[List[int], int]:
    offs, cur = [], 0
    for n in sizes:
        offs.append(cur)
        cur += (int(n) + align - 1) // align * align
    return offs, max(cur, align)


def make_adamw_state(shapes, seed: int, device, grad_dtype=torch.bfloat16,
                     copy_dtype=torch.bfloat16, grad_std: float = 1e-3,
                     loss_scale: float = 65536.0, theta_std: float = 0.02,
                     align: int = ARENA_ALIGN) -> AdamWState:
    names = [n for n, _ in shapes]
    sizes = [numel(s) for _, s in shapes]
    offs, total = layout(sizes, align)
    dev = torch.device(device)
    theta = torch.zeros(total, dtype=torch.float32, device=dev)
    g = _gen(dev, seed, 1)
    for i, n in enumerate(sizes):
        view = theta.narrow(0, offs[i], n)
        torch.randn(n, generator=g, device=dev, dtype=torch.float32, out=view)
        view.mul_(theta_std)
    m = torch.zeros(total, dtype=torch.float32, device=dev)
    v = torch.zeros(total, dtype=torch.float32, device=dev)
    grad = torch.zeros(total, dtype=grad_dtype, device=dev)
    copy = torch.zeros(total, dtype=copy_dtype, device=dev)
    st = AdamWState(names, sizes, offs, theta, m, v, grad, copy, grad_std,
                    loss_scale, seed)
    fill_grads(st, step=1)
    return st


def fill_grads(st: AdamWState, step: int, chunk: int = 1 << 27) -> None:
    """Write the scaled 16-bit gradient draw for ``step`` into the grad arena."""
    dev = st.grad.device
    g = _gen(dev, st.seed, 1000 + int(step))
    for i, n in enumerate(st.sizes):
        view = st.grad.narrow(0, st.offsets[i], n)
        for s in range(0, n, chunk):
            k = min(chunk, n - s)
            tmp = torch.randn(k, generator=g, device=dev, dtype=torch.float32)
            tmp.mul_(st.grad_std * st.loss_scale)
            view.narrow(0, s, k).copy_(tmp)


# ----------------------------------------------------------------------------- softmax bwd
def softmax_inputs(rows: int, cols: int, dtype, seed: int, device,
                   causal_period: int | None = None, causal_offset: int = 0,
                   chunk_rows: int = 8192):
    """Returns ``(P, dY)`` as row-major [rows, cols] tensors of ``dtype``.  With
    ``causal_period`` row r is open on its first min(cols, r % period + 1 + offset)
    columns and P is exactly 0 on the rest."""
    dev = torch.device(device)
    g = _gen(dev, seed, 2)
    P = torch.empty(rows, cols, dtype=dtype, device=dev)
    dY = torch.empty(rows, cols, dtype=dtype, device=dev)
    col = torch.arange(cols, device=dev)
    for r0 in range(0, rows, chunk_rows):
        k = min(chunk_rows, rows - r0)
        z = torch.randn(k, cols, generator=g, device=dev, dtype=torch.float64)
        if causal_period:
            q = (torch.arange(r0, r0 + k, device=dev) % causal_period).unsqueeze(1)
            z = z.masked_fill(col.unsqueeze(0) > q + causal_offset, float("-inf"))
        z = z - z.max(dim=1, keepdim=True).values
        e = torch.exp(z)
        P[r0:r0 + k] = (e / e.sum(dim=1, keepdim=True)).to(dtype)
        dY[r0:r0 + k] = torch.randn(k, cols, generator=g, device=dev,
                                    dtype=torch.float32).to(dtype)
    return P, dY


# ----------------------------------------------------------------------------- LayerNorm bwd
def layernorm_inputs(rows: int, D: int, dtype, seed: int, device, eps: float = 1e-5,
                     dy_std: float = 1.0, chunk_rows: int = 4096):
    """Returns ``(x, dY, mean, inv_std, gamma)``; x, dY in ``dtype``; the rest fp32."""
    dev = torch.device(device)
    g = _gen(dev, seed, 3)
    x = torch.empty(rows, D, dtype=dtype, device=dev)
    dY = torch.empty(rows, D, dtype=dtype, device=dev)
    mean = torch.empty(rows, dtype=torch.float32, device=dev)
    inv_std = torch.empty(rows, dtype=torch.float32, device=dev)
    gamma = (1.0 + 0.1 * torch.randn(D, generator=g, device=dev,
                                     dtype=torch.float32)).contiguous()
    for r0 in range(0, rows, chunk_rows):
        k = min(chunk_rows, rows - r0)
        xs = torch.randn(k, D, generator=g, device=dev, dtype=torch.float32).to(dtype)
        x[r0:r0 + k] = xs
        xd = xs.to(torch.float64)
        mu = xd.mean(dim=1)
        var = ((xd - mu.unsqueeze(1)) ** 2).mean(dim=1)
        mean[r0:r0 + k] = mu.to(torch.float32)
        inv_std[r0:r0 + k] = (1.0 / torch.sqrt(var + eps)).to(torch.float32)
        dY[r0:r0 + k] = (dy_std * torch.randn(k, D, generator=g, device=dev,
                                              dtype=torch.float32)).to(dtype)
    return x, dY, mean, inv_std, gamma


# ----------------------------------------------------------------------------- RMSNorm bwd
def rmsnorm_inputs(rows: int, D: int, dtype, seed: int, device, eps: float = 1e-5,
                   dy_std: float = 1.0, chunk_rows: int = 4096):
    """Returns ``(x, dY, inv_rms, gamma)``; x, dY in ``dtype``; inv_rms = 1/sqrt(mean(x^2)+eps)
    from the stored x in float64, rounded to fp32; gamma ~ N(1, 0.1) fp32."""
    dev = torch.device(device)
    g = _gen(dev, seed, 4)
    x = torch.empty(rows, D, dtype=dtype, device=dev)
    dY = torch.empty(rows, D, dtype=dtype, device=dev)
    inv_rms = torch.empty(rows, dtype=torch.float32, device=dev)
    gamma = (1.0 + 0.1 * torch.randn(D, generator=g, device=dev,
                                     dtype=torch.float32)).contiguous()
    for r0 in range(0, rows, chunk_rows):
        k = min(chunk_rows, rows - r0)
        xs = torch.randn(k, D, generator=g, device=dev, dtype=torch.float32).to(dtype)
        x[r0:r0 + k] = xs
        xd = xs.to(torch.float64)
        inv_rms[r0:r0 + k] = (1.0 / torch.sqrt((xd * xd).mean(dim=1) + eps)).to(torch.float32)
        dY[r0:r0 + k] = (dy_std * torch.randn(k, D, generator=g, device=dev,
                                              dtype=torch.float32)).to(dtype)
    return x, dY, inv_rms, gamma
