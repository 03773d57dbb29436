"""Seeded synthetic workloads of the Muon step (input generation only).

This module holds no arithmetic of the method: it only lists matrix shapes
and draws seeded random inputs (weights, gradients, momentum buffers), so
that the CUDA path and the CPU oracle receive identical inputs.

Workloads (shapes follow the pages' TinyMLP model -- DMuon "Quick Start",
model.py: gate_proj/up_proj are Linear(d, ff) weights [ff, d], down_proj is
Linear(ff, d) [d, ff] -- and Llama-3 projection shapes):

  tinymlp_d128    4 layers x {gate 512x128, up 512x128, down 128x512};
                  grads and momentum i.i.d. N(0, 1)
  tinymlp_d512    4 layers x {gate 2048x512, up 2048x512, down 512x2048};
                  grads N(0, 1e-2^2) (std 1e-2); momentum starts at zero and
                  three steps run with fresh grads
  llama3_8b       32 layers x {q 4096x4096, k 1024x4096, v 1024x4096,
                  o 4096x4096, gate 14336x4096, up 14336x4096,
                  down 4096x14336} = 224 matrices; grads N(0, 1e-3^2);
                  momentum starts at zero with one warm step
  llama3_8b_1layer  the first layer of llama3_8b alone (7 matrices, 1.6 GB
                  of W/G/M: larger than L2, small enough to profile)
  spiked_4096     64 x 4096x4096; grads N(0, 1) plus a rank-16 spike
                  sum_i s_i u_i v_i^T, u, v orthonormal, s_i log-spaced from
                  1e2 down to 1e-3; momentum zero
  tp_70b_mixed    one 28672x8192 matrix (transposed path) plus 512 matrices
                  of 64x256; grads N(0, 1e-3^2); momentum zero

Weights are drawn U(-1/sqrt(cols), 1/sqrt(cols)) like nn.Linear's default
initialisation.  Every tensor is drawn from its own torch.Generator seeded
from (workload seed, matrix index, role, step), so any subset of matrices
can be regenerated alone and on any device.
"""
import math
from dataclasses import dataclass, field

ROLE_W, ROLE_G, ROLE_M = 0, 1, 2


@dataclass(frozen=True)
class Workload:
    name: str
    shapes: tuple
    grad_std: float
    mom_init: str            # "normal" (N(0,1)) or "zero"
    warm_steps: int          # momentum warm-up steps before the measured one
    spike_rank: int = 0
    seed: int = 1234
    note: str = field(default="", compare=False)


def _tinymlp(d, ff, layers=4):
    out = []
    for _ in range(layers):
        out += [(ff, d), (ff, d), (d, ff)]
    return tuple(out)


def _llama3_8b():
    layer = [(4096, 4096), (1024, 4096), (1024, 4096), (4096, 4096),
             (14336, 4096), (14336, 4096), (4096, 14336)]
    return tuple(layer * 32)


WORKLOADS = {
    "tinymlp_d128": Workload("tinymlp_d128", _tinymlp(128, 512), 1.0, "normal", 0, seed=1235,
                             note="TinyMLP d=128 ff=512, 12 matrices"),
    "tinymlp_d512": Workload("tinymlp_d512", _tinymlp(512, 2048), 1e-2, "zero", 2, seed=1236,
                             note="TinyMLP d=512 ff=2048, 12 matrices, 3rd step"),
    "llama3_8b": Workload("llama3_8b", _llama3_8b(), 1e-3, "zero", 1, seed=1237,
                          note="Llama-3-8B projections, 224 matrices"),
    "llama3_8b_1layer": Workload("llama3_8b_1layer", _llama3_8b()[:7], 1e-3, "zero", 1, seed=1237,
                                 note="one Llama-3-8B layer, 7 matrices (profiling case)"),
    "spiked_4096": Workload("spiked_4096", tuple([(4096, 4096)] * 64), 1.0, "zero", 0,
                            spike_rank=16, seed=1238,
                            note="64 x 4096^2 with rank-16 spike"),
    "tp_70b_mixed": Workload("tp_70b_mixed", tuple([(28672, 8192)] + [(64, 256)] * 512), 1e-3,
                             "zero", 0, seed=1239,
                             note="28672x8192 + 512 x 64x256"),
}


def get(name):
    return WORKLOADS[name]


def _gen(seed, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def _seed(w, index, role, step):
    return ((w.seed * 1000003 + index) * 7 + role) * 1009 + step


def weight(w, index, device="cpu"):
    import torch
    r, c = w.shapes[index]
    b = 1.0 / math.sqrt(c)
    t = torch.empty((r, c), dtype=torch.float32, device=device)
    t.uniform_(-b, b, generator=_gen(_seed(w, index, ROLE_W, 0), device))
    return t


def grad(w, index, step=0, device="cpu"):
    """Gradient of matrix `index` at momentum step `step` (0-based)."""
    import torch
    r, c = w.shapes[index]
    g = _gen(_seed(w, index, ROLE_G, step), device)
    t = torch.randn((r, c), dtype=torch.float32, device=device, generator=g)
    if w.grad_std != 1.0:
        t.mul_(w.grad_std)
    if w.spike_rank:
        k = w.spike_rank
        u, _ = torch.linalg.qr(torch.randn((r, k), dtype=torch.float64, device=device, generator=g))
        v, _ = torch.linalg.qr(torch.randn((c, k), dtype=torch.float64, device=device, generator=g))
        s = torch.logspace(2.0, -3.0, k, dtype=torch.float64, device=device)
        t += ((u * s) @ v.T).to(torch.float32)
    return t


def momentum(w, index, device="cpu"):
    import torch
    r, c = w.shapes[index]
    if w.mom_init == "zero":
        return torch.zeros((r, c), dtype=torch.float32, device=device)
    return torch.randn((r, c), dtype=torch.float32, device=device,
                       generator=_gen(_seed(w, index, ROLE_M, 0), device))

