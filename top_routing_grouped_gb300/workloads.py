"""Seeded synthetic MoE-layer workloads: shapes and input tensors, nothing else.

This module is the only thing the CUDA path and the CPU oracle share.  It holds none of
the method's arithmetic: it only draws Gaussian tensors with the stated scales, in a fixed
order, from a seeded CPU generator, and rounds them to the storage type.

Recipe (the same for every configuration):
  * ``torch.Generator().manual_seed(seed)``; fp32 ``randn`` draws in the order
    x [T,d], W_r [E,d], W1 [E,F,d], W3 [E,F,d], W2 [E,d,F];
  * scales: x ~ N(0,1); W_r, W1, W3 ~ N(0, 1/d); W2 ~ N(0, 1/F) (fan-in scaling);
  * bf16 configurations round each drawn fp32 tensor to bf16 (round to nearest even);
    the oracle receives exactly those rounded values;
  * the skewed configuration adds a per-expert router-logit bias
    b_i = 1.5 * ln(1 / (i + 1)) (Zipf-like, rank = expert index);
  * the large configuration uses router temperature 0.5.
"""
from dataclasses import dataclass, replace
import math

import numpy as np
import torch


@dataclass(frozen=True)
class MoEShape:
    name: str
    T: int          # tokens
    d: int          # d_model
    E: int          # experts
    k: int          # experts chosen per token
    F: int          # d_expert
    dtype: str      # "f32" or "bf16": storage and input type of x and the weights
    tau: float = 1.0
    zipf_bias: bool = False
    renorm: bool = False   # variant: gates renormalised over the k chosen
    note: str = ""

    @property
    def N(self):
        """Routed rows: one per (token, chosen expert)."""
        return self.T * self.k

    @property
    def expert_flops(self):
        """Algorithmic FLOPs of the expert FFNs: 3 GEMMs of 2*N*d*F each."""
        return 6 * self.N * self.d * self.F

    def with_(self, **kw):
        return replace(self, **kw)


SHAPES = {
    "tiny_f32": MoEShape("tiny_f32", T=256, d=128, E=8, k=2, F=256, dtype="f32",
                         note="tiny fp32 layer"),
    "coarse_e8": MoEShape("coarse_e8", T=4096, d=2048, E=8, k=2, F=8192, dtype="bf16",
                          note="coarse experts, granularity 1, near-uniform routing"),
    "fine_e32": MoEShape("fine_e32", T=8192, d=2048, E=32, k=8, F=2048, dtype="bf16",
                         note="fine-grained experts, granularity 4"),
    "skewed_e128": MoEShape("skewed_e128", T=16384, d=2048, E=128, k=8, F=1024, dtype="bf16",
                            zipf_bias=True,
                            note="very sparse, Zipf-biased router, some experts empty"),
    "large_e64": MoEShape("large_e64", T=32768, d=4096, E=64, k=4, F=2048, dtype="bf16",
                          tau=0.5, note="large layer, router temperature 0.5"),
}

# The order the workloads are listed in: tiny fp32, coarse, fine, skewed, large.
ORDER = ["tiny_f32", "coarse_e8", "fine_e32", "skewed_e128", "large_e64"]


def granularity_sweep(T=8192, d=2048, d_ff=8192, base_experts=8, base_k=2, Gs=(1, 2, 4, 8)):
    """Layers of equal active FLOPs and equal total expert parameters that differ only in
    granularity G = d_ff / d_expert ("Compute-Optimal Is Not Cluster-Optimal", the 4-D
    scaling law's G): E = base_experts * G experts of width d_ff / G, top-(base_k * G)."""
    return [MoEShape(f"granularity_g{G}", T=T, d=d, E=base_experts * G, k=base_k * G, F=d_ff // G,
                     dtype="bf16", note=f"granularity G={G}") for G in Gs]


@dataclass
class MoEInputs:
    shape: MoEShape
    x: torch.Tensor          # [T, d]
    w_router: torch.Tensor   # [E, d]
    bias: torch.Tensor       # [E] fp32 or None
    w1: torch.Tensor         # [E, F, d]
    w3: torch.Tensor         # [E, F, d]
    w2: torch.Tensor         # [E, d, F]

    def to(self, device):
        mv = lambda t: None if t is None else t.to(device, non_blocking=False).contiguous()
        return MoEInputs(self.shape, mv(self.x), mv(self.w_router), mv(self.bias), mv(self.w1),
                         mv(self.w3), mv(self.w2))

    def numpy_for_oracle(self):
        """Host numpy views: fp32 arrays, or uint16 bf16 bit patterns for bf16 shapes."""
        def cv(t):
            if t is None:
                return None
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16)
            return t.numpy()
        return dict(x=cv(self.x), wr=cv(self.w_router), w1=cv(self.w1), w3=cv(self.w3),
                    w2=cv(self.w2),
                    bias=None if self.bias is None else self.bias.detach().cpu().numpy())


def zipf_bias(E):
    """b_i = 1.5 * ln(1/(i+1)) for expert i (natural log), fp32."""
    return torch.tensor([1.5 * math.log(1.0 / (i + 1)) for i in range(E)], dtype=torch.float32)


def make_inputs(shape: MoEShape, seed: int = 0, parts=("x", "wr", "w1", "w3", "w2")):
    """Draw the workload's tensors on the CPU.  ``parts`` may leave out tensors that a
    caller does not need (they are still drawn, so the others keep their values)."""
    g = torch.Generator().manual_seed(seed)
    T, d, E, F = shape.T, shape.d, shape.E, shape.F
    store = torch.bfloat16 if shape.dtype == "bf16" else torch.float32

    def draw(size, std, keep):
        t = torch.randn(*size, generator=g, dtype=torch.float32)
        if not keep:
            return None
        t.mul_(std)
        return t.to(store).contiguous()

    x = draw((T, d), 1.0, "x" in parts)
    wr = draw((E, d), 1.0 / math.sqrt(d), "wr" in parts)
    w1 = draw((E, F, d), 1.0 / math.sqrt(d), "w1" in parts) if "w1" in parts else None
    # W3 and W2 come after W1 in the stream; when W1 was skipped they cannot be drawn
    # without drawing it, so they are only available together with it.
    w3 = draw((E, F, d), 1.0 / math.sqrt(d), "w3" in parts) if "w1" in parts else None
    w2 = draw((E, d, F), 1.0 / math.sqrt(F), "w2" in parts) if "w1" in parts else None
    bias = zipf_bias(E) if shape.zipf_bias else None
    return MoEInputs(shape, x, wr, bias, w1, w3, w2)
