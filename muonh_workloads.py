"""Seeded synthetic inputs for the MuonH optimizer-step workloads.

This module only draws random numbers and lays out shapes; it holds none of
the method's arithmetic.  Tests, the bench and the smoke check draw inputs
here and hand the same tensors to the CUDA library and to the oracle.

Every matrix is drawn from its own ``torch.Generator`` whose seed is a fixed
function of (what is drawn, step, matrix index), so any subset of a workload
can be drawn alone and equals the same matrices of the full draw on the same
device.  Draws on CUDA and on CPU differ (torch uses different generators
there); parity tests therefore copy device draws to the host.

The shapes stand in for the weights of the Qwen3-style decoder named on the
Puro-2B model card (axforge.ai), "Quickstart" and "Training" sections: model
width 2048, 16 query / 8 key-value heads of dim 128, MLP width 6144, 28
layers.  Weights are N(0, 0.02^2); gradients as each workload states.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch

NS_COEFFS = (3.4445, -4.7750, 2.0315)

_KIND_W, _KIND_G = 1, 2


def _seed(kind: int, step: int, index: int) -> int:
    return ((kind * 1_000_003 + step) * 1_000_003 + index) % (2 ** 62)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


@dataclass
class Workload:
    """A named list of matrix shapes plus how its inputs are drawn."""

    name: str
    shapes: list
    grad_kind: str = "normal"          # normal | student_t3 | low_rank8
    w_std: float = 0.02
    g_scale: float = 1e-3
    beta: float = 0.95
    lr: float = 0.02
    ns_steps: int = 5
    coeffs: tuple = NS_COEFFS
    eps: float = 1e-7
    steps: int = 1
    labels: list = field(default_factory=list)

    @property
    def n_params(self) -> int:
        return sum(r * c for r, c in self.shapes)

    def weight(self, i: int, device="cpu") -> torch.Tensor:
        r, c = self.shapes[i]
        g = _gen(device, _seed(_KIND_W, 0, i))
        return torch.randn(r, c, generator=g, device=device, dtype=torch.float32) * self.w_std

    def grad(self, i: int, step: int = 0, device="cpu") -> torch.Tensor:
        r, c = self.shapes[i]
        g = _gen(device, _seed(_KIND_G, step, i))
        kw = dict(generator=g, device=device, dtype=torch.float32)
        if self.grad_kind == "normal":
            return torch.randn(r, c, **kw) * self.g_scale
        if self.grad_kind == "student_t3":
            # Student-t with 3 degrees of freedom: Z / sqrt(chi2_3 / 3),
            # chi2_3 being the sum of three squared standard normals.
            z = torch.randn(r, c, **kw)
            chi = torch.randn(3, r, c, **kw).square().sum(0)
            return z * torch.rsqrt(chi / 3.0) * self.g_scale
        if self.grad_kind == "low_rank8":
            u = torch.randn(r, 8, **kw)
            v = torch.randn(8, c, **kw)
            noise = torch.randn(r, c, **kw) * 1e-5
            prev = torch.backends.cuda.matmul.allow_tf32
            torch.backends.cuda.matmul.allow_tf32 = False
            try:
                return u @ v + noise
            finally:
                torch.backends.cuda.matmul.allow_tf32 = prev
        raise ValueError(self.grad_kind)

    def weights(self, device="cpu", indices=None):
        idx = range(len(self.shapes)) if indices is None else indices
        return [self.weight(i, device) for i in idx]

    def grads(self, step: int = 0, device="cpu", indices=None):
        idx = range(len(self.shapes)) if indices is None else indices
        return [self.grad(i, step, device) for i in idx]


D_MODEL, N_Q, N_KV, HEAD_DIM, D_FF, N_LAYERS = 2048, 16, 8, 128, 6144, 28

LAYER_SHAPES = [
    (N_Q * HEAD_DIM, D_MODEL),    # Wq
    (N_KV * HEAD_DIM, D_MODEL),   # Wk
    (N_KV * HEAD_DIM, D_MODEL),   # Wv
    (D_MODEL, N_Q * HEAD_DIM),    # Wo
    (D_FF, D_MODEL),              # gate
    (D_FF, D_MODEL),              # up
    (D_MODEL, D_FF),              # down
]
LAYER_LABELS = ["q", "k", "v", "o", "gate", "up", "down"]


def single_256x128() -> Workload:
    """One 256x128 matrix, one step."""
    return Workload("single_256x128", [(256, 128)], labels=["w"])


def qwen3_layer() -> Workload:
    """The seven matrices of one decoder layer (width 2048, GQA 16/8x128, MLP 6144)."""
    return Workload("qwen3_layer_d2048", list(LAYER_SHAPES), labels=list(LAYER_LABELS))


def qwen3_2b(steps: int = 10, layers: int = N_LAYERS) -> Workload:
    """28 layers of decoder matrices: 196 matrices, 1.409 G parameters.

    `layers` < 28 gives the first layers of the same set (same seeds), a
    smaller case with the same bucket shapes for profiling."""
    shapes, labels = [], []
    for layer in range(layers):
        shapes += LAYER_SHAPES
        labels += [f"{layer}.{n}" for n in LAYER_LABELS]
    name = "qwen3_2b_28layers" if layers == N_LAYERS else f"qwen3_2b_first{layers}layers"
    return Workload(name, shapes, steps=steps, labels=labels)


def batched_256(count: int = 1024) -> Workload:
    """``count`` independent 256x256 matrices with heavy-tailed gradients."""
    return Workload(f"batched_{count}x256x256", [(256, 256)] * count,
                    grad_kind="student_t3",
                    labels=[str(i) for i in range(count)])


def aspect_16384x1024() -> Workload:
    """Four 16384x1024 and four 1024x16384 matrices with rank-8 gradients."""
    shapes = [(16384, 1024)] * 4 + [(1024, 16384)] * 4
    return Workload("aspect_16384x1024", shapes, grad_kind="low_rank8",
                    labels=[f"tall{i}" for i in range(4)] + [f"wide{i}" for i in range(4)])


def adamw_group() -> Workload:
    """The parameters outside the MuonH group of a Qwen3-style 2B model, for
    AdamW: a token embedding of 151936 x 2048 (the pages give no vocabulary
    size; this is the Qwen3 family's), two RMSNorm weights per layer and the
    final one (57 x 2048), and the q/k head norms (56 x 128).  Vectors are
    1 x n matrices here.  lr 2e-3 is the MuonH rate divided by the model
    card's 10x multiplier."""
    shapes = [(151936, D_MODEL)] + [(1, D_MODEL)] * (2 * N_LAYERS + 1) + [(1, HEAD_DIM)] * (2 * N_LAYERS)
    return Workload("qwen3_2b_adamw_group", shapes, lr=2e-3, g_scale=1e-2)


ALL = {
    "single_256x128": single_256x128,
    "qwen3_layer_d2048": qwen3_layer,
    "qwen3_2b_28layers": qwen3_2b,
    "batched_1024x256x256": batched_256,
    "aspect_16384x1024": aspect_16384x1024,
    "qwen3_2b_adamw_group": adamw_group,
}


def ragged(shapes, grad_kind="normal", name="ragged") -> Workload:
    """A custom list of shapes (used for tile-tail and edge-case tests)."""
    return Workload(name, list(shapes), grad_kind=grad_kind,
                    labels=[f"{r}x{c}" for r, c in shapes])
