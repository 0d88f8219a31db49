"""Seeded synthetic inputs for the sparse MoE expert block.

This module draws random tensors and nothing else: it holds none of the
block's arithmetic (no routing, no sort, no GEMM, no combine).  Both the CUDA
path and the CPU oracle are fed from here, so that the two sides see
bit-identical inputs.

Workloads (all synthetic; the pages name no dataset):

* ``tiny_fwd``: T=256, emb=256, E=8, top_k=2, mlp=512, softmax over the two
  selected logits.
* ``token_sweep_T{1024,2048,4096,8192}``: emb=2048, E=128, top_k=8, mlp=768,
  softmax-renormalised top-8 weights (the fused-MoE token sweep of the vLLM
  TPU "Fused MoE Kernel integration and optimization" page, benchmark table).
* ``long_seq_train``: T=32768 (2 x 16384), emb=2816, E=128, top_k=8, mlp=704,
  router logits plus a per-expert bias (the Gemma4-26B-A4B workload of the
  MaxText "fused TensorCore Pallas permute/combine kernels" page, Context:
  128 experts, top-8, seq 16k, batch 2; wi = 128*2816*1408*2 B ~ 1 GB).
* ``large_expert_train``: T=8192, emb=7168, E=256, top_k=8, mlp=2048,
  sigmoid scores normalised to sum 1.
* ``zipf_skew_train``: T=16384, emb=2048, E=128, top_k=8, mlp=768; ids drawn
  without replacement from Zipf(1.2) over experts, weights Dirichlet(1).

Value distributions: activations x and the output gradient dy ~ N(0,1);
weights wi, wo ~ N(0, 0.02) (0.02 is the standard deviation); router logits
fp32 ~ N(0,1); bias ~ N(0, 0.5).  Every bf16 tensor is drawn in fp32 and
rounded to bf16 by round-to-nearest-even.  Seed 0 unless stated.  The draw
order is fixed: logits, bias, x, wi (one expert at a time), wo (one expert at
a time), dy.  The Zipf/Dirichlet routing of ``zipf_skew_train`` is drawn on
the host with numpy's PCG64.
"""
from __future__ import annotations

from dataclasses import dataclass, field, asdict

import numpy as np
import torch

SCORE_SOFTMAX_TOPK = 0
SCORE_SIGMOID_NORM = 1
SCORE_GIVEN = 2


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    D: int
    E: int
    K: int
    F: int
    score_mode: int = SCORE_SOFTMAX_TOPK
    bias_std: float = 0.0          # 0 -> no per-expert bias
    zipf_s: float = 0.0            # >0 -> host-drawn Zipf ids, Dirichlet weights
    train: bool = False            # True -> forward + backward
    seed: int = 0

    @property
    def R(self) -> int:
        return self.T * self.K

    def dims(self) -> dict:
        return dict(T=self.T, D=self.D, E=self.E, K=self.K, F=self.F)

    def describe(self) -> dict:
        d = asdict(self)
        d["R"] = self.R
        return d


WORKLOADS: dict[str, Workload] = {
    "tiny_fwd": Workload("tiny_fwd", 256, 256, 8, 2, 512),
    **{
        f"token_sweep_T{t}": Workload(f"token_sweep_T{t}", t, 2048, 128, 8, 768)
        for t in (1024, 2048, 4096, 8192)
    },
    "long_seq_train": Workload("long_seq_train", 32768, 2816, 128, 8, 704,
                               bias_std=0.5, train=True),
    "large_expert_train": Workload("large_expert_train", 8192, 7168, 256, 8, 2048,
                                   score_mode=SCORE_SIGMOID_NORM, train=True),
    "zipf_skew_train": Workload("zipf_skew_train", 16384, 2048, 128, 8, 768,
                                score_mode=SCORE_GIVEN, zipf_s=1.2, train=True),
}


def custom(name: str = "custom", **kw) -> Workload:
    """A workload with explicit sizes (used by tests for small and edge cases)."""
    return Workload(name=name, **kw)


def _normal(shape, std, gen, device, out_dtype):
    t = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(out_dtype)


def zipf_routing(T: int, E: int, K: int, s: float, seed: int):
    """Expert ids drawn without replacement from p(e) ~ (e+1)^-s, K per token,
    by Gumbel-top-k on log p (equivalent to successive sampling without
    replacement); weights ~ Dirichlet(1) over the K slots, fp32.

    Returns (ids int32 [T,K], w float32 [T,K]) as numpy arrays."""
    rng = np.random.Generator(np.random.PCG64(seed))
    logp = -s * np.log(np.arange(1, E + 1, dtype=np.float64))
    gumbel = -np.log(-np.log(rng.random((T, E))))
    keys = logp[None, :] + gumbel
    ids = np.argsort(-keys, axis=1, kind="stable")[:, :K].astype(np.int32)
    w = rng.dirichlet(np.ones(K), size=T).astype(np.float32)
    return np.ascontiguousarray(ids), np.ascontiguousarray(w)


def make_inputs(wl: Workload, device="cpu", *, with_grad: bool | None = None) -> dict:
    """Draw every input of one step of the block for workload ``wl``.

    Returns a dict of torch tensors on ``device``:
      logits fp32 [T,E] (None when routing is given), bias fp32 [E] or None,
      x bf16 [T,D], wi bf16 [E,D,2F], wo bf16 [E,F,D], dy bf16 [T,D] (when
      ``with_grad``), ids int32 [T,K] and w fp32 [T,K] (given routing only).
    """
    if with_grad is None:
        with_grad = wl.train
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed)
    T, D, E, K, F = wl.T, wl.D, wl.E, wl.K, wl.F
    out: dict = {"workload": wl}
    if wl.score_mode == SCORE_GIVEN:
        out["logits"] = None
    else:
        out["logits"] = _normal((T, E), 1.0, gen, device, torch.float32)
    out["bias"] = (_normal((E,), wl.bias_std, gen, device, torch.float32)
                   if wl.bias_std > 0 else None)
    out["x"] = _normal((T, D), 1.0, gen, device, torch.bfloat16)
    wi = torch.empty((E, D, 2 * F), dtype=torch.bfloat16, device=device)
    for e in range(E):
        wi[e] = _normal((D, 2 * F), 0.02, gen, device, torch.bfloat16)
    wo = torch.empty((E, F, D), dtype=torch.bfloat16, device=device)
    for e in range(E):
        wo[e] = _normal((F, D), 0.02, gen, device, torch.bfloat16)
    out["wi"], out["wo"] = wi, wo
    out["dy"] = _normal((T, D), 1.0, gen, device, torch.bfloat16) if with_grad else None
    if wl.score_mode == SCORE_GIVEN:
        if wl.zipf_s > 0:
            ids, w = zipf_routing(T, E, K, wl.zipf_s, wl.seed)
        else:
            rng = np.random.Generator(np.random.PCG64(wl.seed))
            ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
            w = rng.dirichlet(np.ones(K), size=T).astype(np.float32)
        out["ids"] = torch.from_numpy(ids).to(device)
        out["w"] = torch.from_numpy(w).to(device)
    else:
        out["ids"] = None
        out["w"] = None
    return out


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a CPU/GPU bf16 tensor as a numpy uint16 array."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bits_to_bf16(a: np.ndarray) -> torch.Tensor:
    """Inverse of :func:`bf16_bits`."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
