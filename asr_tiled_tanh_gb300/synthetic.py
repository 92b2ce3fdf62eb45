"""Seeded synthetic inputs for the RNN-T joint/output/loss path.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic, so the CUDA library and the CPU oracle can both be fed
from it without sharing any computation.

The workloads stand in for the ones the pages measure on (a 114M-parameter
ASR model on unnamed data in the Flash RNN-T blog, "What changed in practice";
batch 1024 at 40 s of audio in the sample-wise paper's abstract and
conclusion), which are not available.  Shapes and distributions:

  name     B     T    U  HA=HL=H  V      dtype  lengths (uniform, inclusive)        labels
  tiny     2     32   8    64     32     fp32   full                                uniform 1..V-1
  small    8     200  50   512    1024   bf16   T in [T/2,T],   U in [U/2,U]        uniform 1..V-1
  audio20  32    500  100  640    1024   bf16   [0.5,1.0] x max                     uniform 1..V-1
  bigvocab 16    400  80   1024   16384  bf16   [0.5,1.0] x max                     Zipf s=1.1 over 1..V-1
  audio40  1024  1000 100  512    4096   bf16   T in [0.3T,T],  U in [0.3U,U]       uniform 1..V-1

hA, hL ~ N(0,1); W^A ~ N(0,1/HA), W^L ~ N(0,1/HL), W^O ~ N(0,1/H); biases are
zero unless ``bias_std`` is given.  Values are drawn in fp32 and rounded to
bf16 (round to nearest even) for the bf16 workloads.  Draw order: lengths,
labels, hA, hL, W^A, W^L, W^O, b^Z, b^O.  Sample 0 always gets the full
(T, U) so the padded edges of every other sample and the full extent are both
exercised.  Integer ranges run from ceil(frac * max) to max inclusive.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BLANK = 0


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    U: int            # label sequence length; the lattice has U+1 label positions
    HA: int
    HL: int
    H: int
    V: int
    dtype: str        # "f32" or "bf16"
    t_frac: float     # T_len drawn uniformly from [ceil(t_frac*T), T]
    u_frac: float
    labels: str       # "uniform" or "zipf1.1"
    seed: int

    @property
    def U1(self) -> int:
        return self.U + 1

    @property
    def nominal_cells(self) -> int:
        return self.B * self.T * self.U1


WORKLOADS = {
    "tiny": Workload("tiny", 2, 32, 8, 64, 64, 64, 32, "f32", 1.0, 1.0, "uniform", 0),
    "small": Workload("small", 8, 200, 50, 512, 512, 512, 1024, "bf16", 0.5, 0.5, "uniform", 1),
    "audio20": Workload("audio20", 32, 500, 100, 640, 640, 640, 1024, "bf16", 0.5, 0.5,
                        "uniform", 2),
    "bigvocab": Workload("bigvocab", 16, 400, 80, 1024, 1024, 1024, 16384, "bf16", 0.5, 0.5,
                         "zipf1.1", 3),
    "audio40": Workload("audio40", 1024, 1000, 100, 512, 512, 512, 4096, "bf16", 0.3, 0.3,
                        "uniform", 4),
}


@dataclass
class Inputs:
    """Host tensors (torch, CPU).  Float tensors have the workload's dtype."""
    wl: Workload
    hA: torch.Tensor      # [B,T,HA]
    hL: torch.Tensor      # [B,U1,HL]
    WA: torch.Tensor      # [H,HA]
    WL: torch.Tensor      # [H,HL]
    bZ: torch.Tensor      # [H]
    WO: torch.Tensor      # [V,H]
    bO: torch.Tensor      # [V]
    labels: torch.Tensor  # [B,U1] int32, column 0 = blank
    T_len: torch.Tensor   # [B] int32
    U_len: torch.Tensor   # [B] int32
    extra: dict = field(default_factory=dict)

    @property
    def torch_dtype(self):
        return torch.float32 if self.wl.dtype == "f32" else torch.bfloat16

    def valid_cells(self) -> int:
        return int((self.T_len.long() * (self.U_len.long() + 1)).sum())

    def subset(self, idx) -> "Inputs":
        """The same tensors restricted to the samples ``idx`` (a sub-batch)."""
        idx = torch.as_tensor(idx, dtype=torch.long)
        wl = Workload(self.wl.name + "-sub", len(idx), self.wl.T, self.wl.U, self.wl.HA,
                      self.wl.HL, self.wl.H, self.wl.V, self.wl.dtype, self.wl.t_frac,
                      self.wl.u_frac, self.wl.labels, self.wl.seed)
        return Inputs(wl, self.hA[idx].contiguous(), self.hL[idx].contiguous(), self.WA, self.WL,
                      self.bZ, self.WO, self.bO, self.labels[idx].contiguous(),
                      self.T_len[idx].contiguous(), self.U_len[idx].contiguous())


def _lengths(g, n, lo_frac, hi):
    lo = max(1 if hi > 0 else 0, math.ceil(lo_frac * hi))
    return torch.randint(lo, hi + 1, (n,), generator=g, dtype=torch.int64)


def _zipf_probs(V: int, s: float) -> torch.Tensor:
    ranks = torch.arange(1, V, dtype=torch.float64)
    p = ranks.pow(-s)
    return p / p.sum()


def make(wl: Workload | str, seed: int | None = None, bias_std: float = 0.0,
         full_first: bool = True) -> Inputs:
    """Draw the inputs of a workload (CPU, seeded, deterministic)."""
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    g = torch.Generator().manual_seed(wl.seed if seed is None else seed)
    B, T, U1 = wl.B, wl.T, wl.U1
    # lengths
    T_len = _lengths(g, B, wl.t_frac, T)
    U_len = _lengths(g, B, wl.u_frac, wl.U) if wl.U > 0 else torch.zeros(B, dtype=torch.int64)
    if full_first and B > 0:
        T_len[0], U_len[0] = T, wl.U
    # labels (column 0 is the prepended blank)
    if wl.labels == "uniform":
        lab = torch.randint(1, wl.V, (B, U1), generator=g, dtype=torch.int64)
    elif wl.labels.startswith("zipf"):
        s = float(wl.labels[4:])
        p = _zipf_probs(wl.V, s)
        lab = torch.multinomial(p, B * U1, replacement=True, generator=g).view(B, U1) + 1
    else:
        raise ValueError(wl.labels)
    lab[:, 0] = BLANK
    # values, fp32 then rounded to the workload dtype
    f = torch.float32
    hA = torch.randn(B, T, wl.HA, generator=g, dtype=f)
    hL = torch.randn(B, U1, wl.HL, generator=g, dtype=f)
    WA = torch.randn(wl.H, wl.HA, generator=g, dtype=f) / math.sqrt(wl.HA)
    WL = torch.randn(wl.H, wl.HL, generator=g, dtype=f) / math.sqrt(wl.HL)
    WO = torch.randn(wl.V, wl.H, generator=g, dtype=f) / math.sqrt(wl.H)
    if bias_std > 0:
        bZ = torch.randn(wl.H, generator=g, dtype=f) * bias_std
        bO = torch.randn(wl.V, generator=g, dtype=f) * bias_std
    else:
        bZ = torch.zeros(wl.H, dtype=f)
        bO = torch.zeros(wl.V, dtype=f)
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    cast = lambda x: x.to(dt).contiguous()
    return Inputs(wl, cast(hA), cast(hL), cast(WA), cast(WL), cast(bZ), cast(WO), cast(bO),
                  lab.to(torch.int32).contiguous(), T_len.to(torch.int32).contiguous(),
                  U_len.to(torch.int32).contiguous())


def custom(B, T, U, HA, HL, H, V, dtype="f32", seed=0, t_frac=0.5, u_frac=0.5,
           labels="uniform", bias_std=0.0, full_first=True) -> Inputs:
    """Inputs of an ad-hoc shape with the same value distributions."""
    wl = Workload(f"custom-B{B}T{T}U{U}H{H}V{V}", B, T, U, HA, HL, H, V, dtype, t_frac, u_frac,
                  labels, seed)
    return make(wl, bias_std=bias_std, full_first=full_first)
