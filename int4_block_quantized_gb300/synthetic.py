"""Seeded synthetic inputs for the INT4 block-quantized MoE FFN layer.

This module only draws random numbers in the layouts the library and the
oracle consume; it holds none of the layer's arithmetic.  Both the CUDA
path's tests/bench and the fp64 oracle receive the same tensors from here.

Layouts (all contiguous):
  x          [T, H]        fp16 or bf16 activations
  router_w   [H, E]        same dtype as x
  router_bias[E]           fp32 or None
  gate_w/up_w[E, I, H/2]   uint8, two uint4 per byte, low nibble = even k
  gate_s/up_s[E, I, H/bs]  fp16 or bf16 block scales
  gate_zp/.. [E, I, H/bs]  uint8 zero points 0..15, or None (zero point 8)
  down_w     [E, H, I/2], down_s / down_zp [E, H, I/bs]

Distributions per workload (see WORKLOADS): uint4 codes uniform on 0..15
(each byte is uniform on 0..255, i.e. two independent uniform nibbles),
scales uniform[0.5, 1.5] * 2^-5 (fp16) or * 2^-6 (bf16), zero points
uniform on 0..15, x ~ N(0, 1), router_w ~ N(0, 0.02).  The prefill workload
skews routing with a Zipf(s=1.1) per-expert logit bias
b_e = ln(r_e^-s / sum_{r=1..E} r^-s), r_e = 1 + pi(e) for a seeded
permutation pi.

Every tensor has its own generator seeded with
seed*1000 + tensor_id + 100000*layer, so a tensor does not change when
another one's shape does.
"""
import math
from dataclasses import dataclass, replace
from typing import Optional

import torch

F16, BF16 = 0, 1
_TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16}

_TID = {"x": 0, "router_w": 1, "router_bias": 2,
        "gate_w": 3, "gate_s": 4, "gate_zp": 5,
        "up_w": 6, "up_s": 7, "up_zp": 8,
        "down_w": 9, "down_s": 10, "down_zp": 11,
        "shared_sg": 12,
        "shared_gate_w": 13, "shared_gate_s": 14, "shared_gate_zp": 15,
        "shared_up_w": 16, "shared_up_s": 17, "shared_up_zp": 18,
        "shared_down_w": 19, "shared_down_s": 20, "shared_down_zp": 21}


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    block_size: int
    act_dtype: int
    scale_dtype: int
    has_zp: bool
    scale_exp: int          # scales ~ U[0.5, 1.5] * 2^scale_exp
    zipf_s: float = 0.0     # 0 = no router bias
    layers: int = 1
    router_std: float = 0.02
    x_std: float = 1.0

    def with_(self, **kw):
        return replace(self, **kw)


WORKLOADS = {
    # T=4, H=256, I=128, E=8, k=2, uint4 zero points, fp16 scales/activations, seed 0
    "tiny": Workload("tiny", 4, 256, 128, 8, 2, 32, F16, F16, True, -5),
    # Qwen1.5-MoE-A2.7B-shaped decode layer, one token
    "decode": Workload("decode", 1, 2048, 1408, 60, 4, 32, F16, F16, True, -5),
    # same layer, a 16-token speculative-verify batch
    "verify": Workload("verify", 16, 2048, 1408, 60, 4, 32, F16, F16, True, -5),
    # 512-token prefill, signed symmetric int4 (no zero-point tensor), block 128,
    # bf16 scales, Zipf(1.1)-skewed routing
    "prefill": Workload("prefill", 512, 2048, 1408, 60, 4, 128, BF16, BF16, False, -6, zipf_s=1.1),
    # 24-layer residual stack x += layer(RMSNorm(x)), 2048 tokens
    "stack": Workload("stack", 2048, 2048, 1408, 60, 4, 32, BF16, F16, True, -5, layers=24),
    # larger-E members of the family: 128 experts, top-8, I = 768 and
    # 256 experts, top-8, I = 512 (H = 2048), decode and prefill batches
    "e128_decode": Workload("e128_decode", 1, 2048, 768, 128, 8, 32, F16, F16, True, -5),
    "e128_prefill": Workload("e128_prefill", 512, 2048, 768, 128, 8, 128, BF16, BF16, False, -6),
    "e256_decode": Workload("e256_decode", 1, 2048, 512, 256, 8, 32, F16, F16, True, -5),
    "e256_prefill": Workload("e256_prefill", 512, 2048, 512, 256, 8, 128, BF16, BF16, False, -6),
    # shared expert of the Qwen1.5-MoE-A2.7B block (intermediate 5632 = 4 x 1408),
    # in the same INT4 block format; E = k = 1 (make_shared_expert)
    "shared_decode": Workload("shared_decode", 1, 2048, 5632, 1, 1, 32, F16, F16, True, -5),
    "shared_prefill": Workload("shared_prefill", 512, 2048, 5632, 1, 1, 128, BF16, BF16, False, -6),
}


def _gen(device, seed, layer, name):
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + _TID[name] + 100000 * layer)
    return g


def zipf_bias(E: int, s: float, perm: torch.Tensor) -> torch.Tensor:
    """Per-expert logit bias making the routing prior Zipf(s) over a permuted rank."""
    z = sum((r ** -s) for r in range(1, E + 1))
    b = [math.log(((1 + int(perm[e])) ** -s) / z) for e in range(E)]
    return torch.tensor(b, dtype=torch.float64).to(torch.float32)


def make_x(wl: Workload, seed: int = 0, device="cpu", T: Optional[int] = None, layer: int = 0):
    T = wl.T if T is None else T
    g = _gen(device, seed, layer, "x")
    x = torch.randn((T, wl.H), generator=g, device=device, dtype=torch.float32) * wl.x_std
    return x.to(_TORCH_DTYPE[wl.act_dtype])


def _qweight(wl, seed, layer, device, prefix, N, K):
    E, bs = wl.E, wl.block_size
    gw = _gen(device, seed, layer, prefix + "_w")
    w = torch.randint(0, 256, (E, N, K // 2), generator=gw, device=device, dtype=torch.uint8)
    gs = _gen(device, seed, layer, prefix + "_s")
    s = (torch.rand((E, N, K // bs), generator=gs, device=device, dtype=torch.float32) + 0.5)
    s = (s * (2.0 ** wl.scale_exp)).to(_TORCH_DTYPE[wl.scale_dtype])
    zp = None
    if wl.has_zp:
        gz = _gen(device, seed, layer, prefix + "_zp")
        zp = torch.randint(0, 16, (E, N, K // bs), generator=gz, device=device, dtype=torch.uint8)
    return w, s, zp


def make_weights(wl: Workload, seed: int = 0, device="cpu", layer: int = 0) -> dict:
    """One layer's router and expert tensors (no activations)."""
    d = {}
    g = _gen(device, seed, layer, "router_w")
    rw = torch.randn((wl.H, wl.E), generator=g, device=device, dtype=torch.float32) * wl.router_std
    d["router_w"] = rw.to(_TORCH_DTYPE[wl.act_dtype])
    d["router_bias"] = None
    if wl.zipf_s > 0:
        gp = _gen("cpu", seed, layer, "router_bias")
        perm = torch.randperm(wl.E, generator=gp)
        d["router_bias"] = zipf_bias(wl.E, wl.zipf_s, perm).to(device)
    for p, (N, K) in (("gate", (wl.I, wl.H)), ("up", (wl.I, wl.H)), ("down", (wl.H, wl.I))):
        w, s, zp = _qweight(wl, seed, layer, device, p, N, K)
        d[p + "_w"], d[p + "_s"], d[p + "_zp"] = w, s, zp
    d.update(H=wl.H, I=wl.I, E=wl.E, k=wl.k, block_size=wl.block_size,
             act_dtype=wl.act_dtype, scale_dtype=wl.scale_dtype)
    return d


def make_layer(wl: Workload, seed: int = 0, device="cpu", layer: int = 0, T: Optional[int] = None) -> dict:
    """Activations plus one layer's weights, as the dict both sides consume."""
    d = make_weights(wl, seed, device, layer)
    d["x"] = make_x(wl, seed, device, T=T, layer=layer)
    d["T"] = d["x"].shape[0]
    return d


def make_shared_expert(wl: Workload, seed: int = 0, device="cpu", layer: int = 0,
                       T: Optional[int] = None) -> dict:
    """A shared expert: gate vector shared_gate_w [H] (x's dtype, ~N(0, router
    std)) and one expert's gate/up/down tensors ([1, I, H/2], [1, H, I/2]),
    plus activations; keys as in make_layer so the same consumers apply."""
    d = {}
    g = _gen(device, seed, layer, "shared_sg")
    sg = torch.randn((wl.H,), generator=g, device=device, dtype=torch.float32) * wl.router_std
    d["shared_gate_w"] = sg.to(_TORCH_DTYPE[wl.act_dtype])
    one = wl.with_(E=1)
    for p, (N, K) in (("gate", (wl.I, wl.H)), ("up", (wl.I, wl.H)), ("down", (wl.H, wl.I))):
        w, s, zp = _qweight(one, seed, layer, device, "shared_" + p, N, K)
        d[p + "_w"], d[p + "_s"], d[p + "_zp"] = w, s, zp
    d.update(H=wl.H, I=wl.I, E=1, k=1, block_size=wl.block_size,
             act_dtype=wl.act_dtype, scale_dtype=wl.scale_dtype)
    d["x"] = make_x(wl, seed, device, T=T, layer=layer)
    d["T"] = d["x"].shape[0]
    return d


def expert_bytes(wl: Workload) -> int:
    """Bytes of one expert's gate+up+down: packed int4 + scales + zero points."""
    el = 3 * wl.H * wl.I
    blocks = el // wl.block_size
    return el // 2 + blocks * 2 + (blocks if wl.has_zp else 0)
