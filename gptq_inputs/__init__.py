"""Seeded synthetic inputs shaped like Llama-class layers, for tests and benchmarks.

This module only draws random numbers: fp32 weights ~ N(0, 0.02), per-(group, column)
shifts, outlier positions, the act-order row permutation and fp32 activations ~ N(0, 1)
cast to fp16/bf16.  It holds none of the GPTQ arithmetic -- no quantizer, packer or
dequantizer -- so the CPU oracle and the CUDA library can both take their inputs from it
without sharing any of the method's code.  Turning the weights into a packed checkpoint is
the job of the consumer (the oracle's round-to-nearest writer in the tests, the library's
GPU quantizer in the benchmark).

Workloads (the shapes of the layers the pages talk about; their datasets are not needed
and not present -- these seeded draws stand in for them):

  tiny_4bit_g64             A fp16 [4, 512],   W [512, 512]     4-bit, group 64,  v2 and v1
  llama7b_decode_4bit_g128  A fp16 [M, 4096],  W [4096, 11008]  4-bit, group 128, v2 and v1,
                            M in {1, 8, 16}
  lowbit_2bit_g64           A bf16 [M, 4096],  W [4096, 4096]   2-bit, group 64,  v2,
                            M in {1, 8, 32}; each (group, column) shifted by U(-0.064, 0.064)
                            so that the stored zeros span the whole 2-bit range
  act_order_3bit_g128       A fp16 [16, 5120], W [5120, 13824]  3-bit, group 128, v2, 0.5% of
                            entries scaled x20 (outliers), g_idx[k] = perm(k) // 128
  prefill_4bit_g128         A bf16 [4096, 4096], W [4096, 14336] 4-bit, group 128, v2
  prefill_8bit_sym_g128     same A and W, 8-bit symmetric (zero 128), group 128
  prefill_4bit_gall         same A and W, 4-bit, one group per column (group = -1)

Seeds: the weights of a workload use numpy default_rng(seed); activations with M rows use
default_rng(seed * 100 + M).  Draw order inside a seed: W, then shifts, then outlier
positions, then the act-order permutation.

Mixture-of-experts workloads (MOE_WORKLOADS; the grouped GEMM):

  moe_mixtral_4bit_g128     E = 8 experts, each W [4096, 14336] 4-bit, group 128, v2 (the
                            expert up-projection shape of a Mixtral-8x7B-class model); A fp16;
                            T tokens in {1, 8}, each routed to 2 distinct experts

Expert e's weights use default_rng(seed * 1000 + e); the routing of T tokens uses
default_rng(seed * 100 + T) (each token draws its top-k experts without replacement), and the
token activations default_rng(seed * 100 + T + 50).  Rows of the grouped A are the
(token, expert) pairs sorted by expert, then by token.
"""
from dataclasses import dataclass, field, replace
from typing import Optional, Tuple

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    K: int
    N: int
    bits: int
    group: int                 # -1: one group spanning all K rows
    act_dtype: str             # "f16" or "bf16"
    Ms: Tuple[int, ...]
    fmts: Tuple[str, ...]      # "v2", "v1"
    seed: int
    sym: bool = False
    shift: float = 0.0         # half-width of the per-(group, column) uniform shift
    outlier_frac: float = 0.0
    outlier_mult: float = 20.0
    act_order: bool = False

    @property
    def G(self) -> int:
        return 1 if self.group == -1 else self.K // self.group

    def resized(self, K: int, N: int, Ms: Tuple[int, ...], name: Optional[str] = None):
        """Same recipe at another size (used for oracle-sized parity cases)."""
        return replace(self, K=K, N=N, Ms=tuple(Ms), name=name or "%s@%dx%d" % (self.name, K, N))


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_4bit_g64", 512, 512, 4, 64, "f16", (4,), ("v2", "v1"), seed=0),
        Workload("llama7b_decode_4bit_g128", 4096, 11008, 4, 128, "f16", (1, 8, 16),
                 ("v2", "v1"), seed=2),
        Workload("lowbit_2bit_g64", 4096, 4096, 2, 64, "bf16", (1, 8, 32), ("v2",), seed=3,
                 shift=0.064),
        Workload("act_order_3bit_g128", 5120, 13824, 3, 128, "f16", (16,), ("v2",), seed=4,
                 outlier_frac=0.005, act_order=True),
        Workload("prefill_4bit_g128", 4096, 14336, 4, 128, "bf16", (4096,), ("v2",), seed=5),
        Workload("prefill_8bit_sym_g128", 4096, 14336, 8, 128, "bf16", (4096,), ("v2",),
                 seed=5, sym=True),
        Workload("prefill_4bit_gall", 4096, 14336, 4, -1, "bf16", (4096,), ("v2",), seed=5),
    ]
}


@dataclass
class WeightDraw:
    W: np.ndarray                      # fp32 [K, N]
    g_idx: Optional[np.ndarray]        # int32 [K] or None
    shifts: Optional[np.ndarray] = None
    outliers: Optional[np.ndarray] = None


def draw_weights(wl: Workload) -> WeightDraw:
    """fp32 weights [K, N] (and g_idx for act-order workloads), seeded by the workload."""
    rng = np.random.default_rng(wl.seed)
    W = rng.standard_normal((wl.K, wl.N), dtype=np.float32)
    W *= np.float32(0.02)
    shifts = None
    if wl.shift:
        rows_per_group = wl.K if wl.group == -1 else wl.group
        shifts = rng.uniform(-wl.shift, wl.shift, size=(wl.G, wl.N)).astype(np.float32)
        W += np.repeat(shifts, rows_per_group, axis=0)
    outliers = None
    if wl.outlier_frac:
        count = int(round(wl.outlier_frac * wl.K * wl.N))
        outliers = rng.choice(wl.K * wl.N, size=count, replace=False, shuffle=False)
        W.reshape(-1)[outliers] *= np.float32(wl.outlier_mult)
    g_idx = None
    if wl.act_order:
        perm = rng.permutation(wl.K)
        g_idx = (perm // wl.group).astype(np.int32)
    return WeightDraw(W=W, g_idx=g_idx, shifts=shifts, outliers=outliers)


def draw_activations_f32(wl: Workload, M: int) -> np.ndarray:
    rng = np.random.default_rng(wl.seed * 100 + M)
    return rng.standard_normal((M, wl.K), dtype=np.float32)


def draw_activations(wl: Workload, M: int):
    """Activations [M, K] as a CPU torch tensor of the workload's dtype (fp32 draw, RNE cast)."""
    import torch
    a32 = torch.from_numpy(draw_activations_f32(wl, M))
    return a32.to(torch.float16 if wl.act_dtype == "f16" else torch.bfloat16)


def bits16(t) -> np.ndarray:
    """uint16 bit patterns of a CPU fp16/bf16 torch tensor."""
    import torch
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------------ mixture of experts
@dataclass(frozen=True)
class MoeWorkload:
    name: str
    E: int
    K: int
    N: int
    bits: int
    group: int
    act_dtype: str
    Ts: Tuple[int, ...]        # tokens per batch
    topk: int
    seed: int

    @property
    def G(self) -> int:
        return 1 if self.group == -1 else self.K // self.group

    def resized(self, E: int, K: int, N: int, Ts: Tuple[int, ...], name: Optional[str] = None):
        return replace(self, E=E, K=K, N=N, Ts=tuple(Ts), name=name or "%s@%dx%dx%d" % (self.name, E, K, N))


MOE_WORKLOADS = {
    w.name: w for w in [
        MoeWorkload("moe_mixtral_4bit_g128", 8, 4096, 14336, 4, 128, "f16", (1, 8), 2, seed=6),
    ]
}


def draw_expert_weights(mw: MoeWorkload, e: int) -> np.ndarray:
    """fp32 weights [K, N] of expert e."""
    rng = np.random.default_rng(mw.seed * 1000 + e)
    W = rng.standard_normal((mw.K, mw.N), dtype=np.float32)
    W *= np.float32(0.02)
    return W


@dataclass
class Routing:
    row_token: np.ndarray     # int32 [T * topk]: the token of each grouped row
    offsets: np.ndarray       # int32 [E + 1]: rows [offsets[e], offsets[e + 1]) go to expert e


def draw_routing(mw: MoeWorkload, T: int) -> Routing:
    rng = np.random.default_rng(mw.seed * 100 + T)
    experts = np.stack([rng.choice(mw.E, size=mw.topk, replace=False) for _ in range(T)])
    pairs = sorted((int(experts[t, j]), t) for t in range(T) for j in range(mw.topk))
    row_token = np.array([t for _, t in pairs], np.int32)
    counts = np.bincount([e for e, _ in pairs], minlength=mw.E)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return Routing(row_token=row_token, offsets=offsets)


def draw_token_activations(mw: MoeWorkload, T: int):
    """Token activations [T, K] as a CPU torch tensor of the workload's dtype."""
    import torch
    rng = np.random.default_rng(mw.seed * 100 + T + 50)
    a32 = torch.from_numpy(rng.standard_normal((T, mw.K), dtype=np.float32))
    return a32.to(torch.float16 if mw.act_dtype == "f16" else torch.bfloat16)
